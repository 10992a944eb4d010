// Host side of the C ABI declared in include/mhc.h: argument validation,
// the hidden-slice plan, TMA tensor-map encoding and kernel dispatch.
#include <atomic>
#include <chrono>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "mhc.h"
#include "mhc_internal.h"

using namespace mhc;

namespace {

constexpr int kMaxDevices = 64;

std::atomic<unsigned long long> g_timeout_ns{1000000000ull};
thread_local int t_last_site = 0;
thread_local cudaEvent_t t_between_event = nullptr;

struct DeviceInfo {
    std::once_flag once;
    bool ok = false;
    unsigned int *status = nullptr;
    int sms = 0;
};

// Flag value of each shifted call: unique within the process (monotonic),
// started from a time- and address-derived seed so that stale workspace
// contents from another process are not mistaken for this call's flags.
std::atomic<unsigned long long> g_epoch{0};
std::once_flag g_epoch_once;
unsigned long long next_epoch() {
    std::call_once(g_epoch_once, [] {
        const unsigned long long t = static_cast<unsigned long long>(
            std::chrono::high_resolution_clock::now().time_since_epoch().count());
        const unsigned long long a = reinterpret_cast<uintptr_t>(&g_epoch);
        unsigned long long z = t ^ (a << 17) ^ 0x9E3779B97F4A7C15ull;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        g_epoch.store((z ^ (z >> 31)) | 1ull);
    });
    return g_epoch.fetch_add(1) + 1;
}
DeviceInfo g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

mhc_status current_device(DeviceInfo **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MHC_ERR_CUDA;
    DeviceInfo &d = g_dev[dev];
    std::call_once(d.once, [&] {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
            return;
        if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return;
        if (major != 10 || minor != 3) return;   // the library carries sm_103a code only
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return;
        d.status = device_status_word();
        d.ok = d.status != nullptr;
    });
    if (!d.ok) return MHC_ERR_UNSUPPORTED;
    *out = &d;
    return MHC_OK;
}

bool get_encoder() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool hidden_ok(int H) { return H >= kChunk && H <= 65536 && H % kChunk == 0; }

// Half-open byte ranges [a, a + an) and [b, b + bn) intersect.
bool overlap(const void *a, size_t an, const void *b, size_t bn) {
    if (!a || !b || an == 0 || bn == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bn && y < x + an;
}

struct Range {
    const void *p;
    size_t n;
};

// Any output overlapping any input or another output, except an output
// identical (same pointer, same size) to an input marked `may_equal`.
bool aliasing(const Range *outs, int no, const Range *ins, int ni, const void *may_equal_in,
              const void *may_equal_out) {
    for (int i = 0; i < no; ++i) {
        for (int j = 0; j < ni; ++j) {
            if (outs[i].p == may_equal_out && ins[j].p == may_equal_in && outs[i].p == ins[j].p)
                continue;
            if (overlap(outs[i].p, outs[i].n, ins[j].p, ins[j].n)) return true;
        }
        for (int j = i + 1; j < no; ++j)
            if (overlap(outs[i].p, outs[i].n, outs[j].p, outs[j].n)) return true;
    }
    return false;
}

// Hidden-slice plan: items of d chunks (d | H/32; a slice is d interleaved
// 32-wide chunks) spread over kGridCap persistent CTAs. At most kGridCap
// slices, so that every slice of a tile can be in flight at once (the
// shifted form's CTAs wait for one another). Among the item sizes of at most
// 8 chunks (enough CTAs on one tile for DRAM row locality; the shifted
// form's collapse buffer holds 8) minimise the busiest CTA's work, counting
// kItemCost chunks' worth per item for its fixed costs (partials, the
// finishers' waits and reductions). Only when no such size fits, take the
// smallest larger one. A pure function of (T, H), so the workspace size is
// too.
constexpr double kItemCost = 2.0;
constexpr long long kSplitKOneKernelTokens = 1024;
// The batch-invariant plan: a function of H alone, the item size the plan
// converges to for large T (the largest of at most 8 chunks that divides H/32
// with at most kGridCap slices, else the smallest larger one).
void plan_invariant(int H, int *n_slices, int *slice_w) {
    const int chunks = H / kChunk;
    int d = 0;
    for (int c = chunks < 8 ? chunks : 8; c >= 1 && d == 0; --c)
        if (chunks % c == 0 && chunks / c <= kGridCap) d = c;
    if (d == 0) {
        d = 9;
        while (chunks % d || chunks / d > kGridCap) ++d;
    }
    *n_slices = chunks / d;
    *slice_w = d * kChunk;
}

void plan(long long T, int H, int *n_slices, int *slice_w) {
    const int chunks = H / kChunk;
    const long long tiles = (T + kTileT - 1) / kTileT;
    constexpr int kMaxItemChunks = 8;
    double best_cost = -1.0;
    int best_d = 0;
    for (int d = chunks < kMaxItemChunks ? chunks : kMaxItemChunks; d >= 1; --d) {
        if (chunks % d || chunks / d > kGridCap) continue;
        const long long items = tiles * (chunks / d);
        const long long per_cta = (items + kGridCap - 1) / kGridCap;
        const double cost = static_cast<double>(per_cta) * (d + kItemCost);
        if (best_cost < 0 || cost < best_cost - 1e-9) {
            best_cost = cost;
            best_d = d;
        }
    }
    if (best_d == 0) {
        best_d = kMaxItemChunks + 1;
        while (chunks % best_d || chunks / best_d > kGridCap) ++best_d;
    }
    *n_slices = chunks / best_d;
    *slice_w = best_d * kChunk;
}

// Workspace: first a 256-byte area holding the u64 epoch cell that a call
// being captured into a CUDA graph takes its flag value from (at offset 0
// whatever the call's shape, so that calls of different shapes sharing a
// workspace never overwrite it with a flag word, nor read a flag as it),
// then per-item partial blocks [tiles][S] of 128 x 32 fp32, then (each
// 256-byte aligned) the shifted form's per-slice collapse sums [S][T] fp32
// and its publication flags [tiles][S][4] u64.
constexpr size_t kCellBytes = 256;
size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }
size_t partials_bytes(long long T, int S) {
    const size_t tiles = static_cast<size_t>((T + kTileT - 1) / kTileT);
    return align256(tiles * static_cast<size_t>(S) * kItemFloats * sizeof(float));
}
size_t ssql_bytes(long long T, int S) {
    return align256(static_cast<size_t>(S) * static_cast<size_t>(T) * sizeof(float));
}

size_t flags_bytes(long long T, int S) {
    const size_t tiles = static_cast<size_t>((T + kTileT - 1) / kTileT);
    return align256(tiles * static_cast<size_t>(S) * 4 * sizeof(unsigned long long));
}

size_t workspace_layout_bytes(long long T, int S) {
    return kCellBytes + partials_bytes(T, S) + ssql_bytes(T, S) + flags_bytes(T, S);
}

// Enough for the plan of either mode (default and batch-invariant).
size_t workspace_bytes(long long T, int H) {
    if (T <= 0 || !hidden_ok(H)) return 0;
    int S = 0, w = 0, Si = 0, wi = 0;
    plan(T, H, &S, &w);
    plan_invariant(H, &Si, &wi);
    const size_t a = workspace_layout_bytes(T, S), b = workspace_layout_bytes(T, Si);
    return a > b ? a : b;
}

// Token rows per box: a call of one tile loads only the rows it has (rounded
// up to 8), one box per stream; larger calls take whole 128-row tiles of all
// four streams in one box (box_rows 0).
int box_rows_for(long long T) { return T <= kTileT ? static_cast<int>((T + 7) / 8 * 8) : 0; }

// bf16 [rows.., H] viewed by TMA: dim0 = hidden (box 32, 64-byte swizzle).
bool encode_2d(CUtensorMap *m, const void *ptr, int H, long long T) {
    const int br = box_rows_for(T);
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * 2};
    cuuint32_t box[2] = {kChunk, static_cast<cuuint32_t>(br ? br : kTileT)};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [T, 4, H] viewed as (hidden, token, stream) so that a box lands in
// shared memory as [stream][token][32 hidden] (one stream per box when the
// call is a single tile).
bool encode_res(CUtensorMap *m, const void *ptr, int H, long long T, bool all_streams = false) {
    const int br = box_rows_for(T);
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T), 4};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(H) * 8, static_cast<cuuint64_t>(H) * 2};
    cuuint32_t box[3] = {kChunk, static_cast<cuuint32_t>(br ? br : kTileT),
                         br && !all_streams ? 1u : 4u};
    cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps of the last few calls of this host thread, by (kind, pointer,
// H, T) (kind 0 residual-shaped, 1 x-shaped, 2 residual-shaped with the four
// streams in one box of a call's token rows): a decode loop reuses its
// buffers, and encoding costs host time.
struct MapCache {
    struct Entry {
        int kind = -1, H = 0;
        long long T = 0;
        const void *ptr = nullptr;
        CUtensorMap map;
    } e[8];
    int next = 0;
};
thread_local MapCache t_maps;

bool encode_cached(int kind, CUtensorMap *m, const void *ptr, int H, long long T) {
    for (const auto &x : t_maps.e) {
        if (x.kind == kind && x.ptr == ptr && x.H == H && x.T == T) {
            *m = x.map;
            return true;
        }
    }
    const bool ok = kind == 1 ? encode_2d(m, ptr, H, T) : encode_res(m, ptr, H, T, kind == 2);
    if (ok) {
        auto &x = t_maps.e[t_maps.next];
        t_maps.next = (t_maps.next + 1) % 8;
        x.kind = kind;
        x.ptr = ptr;
        x.H = H;
        x.T = T;
        x.map = *m;
    }
    return ok;
}

// Whether the boundary kernels launch as programmatic dependents of the
// previous kernel on the stream (a benchmark hook turns it off).
std::atomic<int> g_pdl{1};

// Decode path of the shifted form: 0 = a cluster where one fits and is the
// faster, 1 = always the slice-parallel streaming kernel, 2 = a cluster
// wherever one fits (test and benchmark hooks).
std::atomic<int> g_decode_path{0};

// Where the cluster kernel is the faster (measured on one box, graph replay
// at 1 to 64 tokens and hidden 512 to 4096 against the slice-parallel
// streaming kernel): when each CTA streams one chunk (by 0.9-2.2 us), two
// chunks for up to 32 tokens (by 0.2-1.7 us), up to four for up to 16 tokens
// (hidden 2048: by 1.0 us at 1 to 8 tokens, 0.25 us at 16). With more chunks
// per CTA its 16 CTAs carry 4-14 times the per-SM work of the slice-parallel
// kernel (weight tiles pulled from L2, elementwise chains, MMA instructions)
// and lose (hidden 4096: even at 1 to 4 tokens, worse from 8).
bool cluster_preferred(long long T, const ClusterArgs &ca) {
    return ca.nch == 1 || (ca.nch == 2 && T <= 32) || (ca.nch <= 4 && T <= 16);
}

// The shifted call of at most kClusterMaxTokens tokens on one thread-block
// cluster: the largest cluster size C <= 16 dividing the H/32 chunks with at
// most kClusterMaxChunks chunks per CTA; stages packed by token rows, as many
// as fit beside the CTA's collapse buffer and the exchange areas (every chunk
// resident when they all fit, else a ring of at least two). False when the
// shape has no such plan.
bool cluster_plan(long long T, int H, ClusterArgs *ca) {
    if (T < 1 || T > kClusterMaxTokens) return false;
    const int chunks = H / kChunk;
    int C = 0;
    for (int c = kClusterMaxCtas; c >= 1 && C == 0; --c)
        if (chunks % c == 0 && chunks / c <= kClusterMaxChunks) C = c;
    if (C == 0) return false;
    const int nch = chunks / C;
    const int R = static_cast<int>((T + 7) / 8 * 8);
    const uint32_t stage = 5u * R * kRowBytes + kWBytes;          // a multiple of 512
    const uint32_t li = static_cast<uint32_t>(nch) * R * kRowBytes;
    const uint32_t owned_max = static_cast<uint32_t>((T + C - 1) / C);
    const uint32_t part = (owned_max * C * kClusterRecFloats * 4 + 15u) & ~15u;
    const uint32_t sql = (static_cast<uint32_t>(C * T) * 4 + 15u) & ~15u;
    const uint32_t red = (16 * kPartVals + 32 + kClusterMaxTokens) * 4;
    const uint32_t misc = 1024 /* alignment of li's end */ + 512 /* barriers */ +
                          8 * 2 * kClusterMaxTokens * 4 + part + sql + red + 1024 /* base alignment */;
    if (li + misc + 2 * stage > static_cast<uint32_t>(kClusterSmemMax) &&
        li + misc + static_cast<uint32_t>(nch) * stage > static_cast<uint32_t>(kClusterSmemMax))
        return false;
    int NS = static_cast<int>((kClusterSmemMax - li - misc) / stage);
    if (NS > nch) NS = nch;
    if (NS > kClusterMaxStages) NS = kClusterMaxStages;
    if (NS < 2 && NS < nch) return false;
    ca->T = static_cast<int>(T);
    ca->H = H;
    ca->ctas = C;
    ca->nch = nch;
    ca->rows = R;
    ca->stages = NS;
    ca->stage_bytes = stage;
    ca->li_off = NS * stage;
    ca->bar_off = (ca->li_off + li + 1023u) & ~1023u;
    ca->sums_off = ca->bar_off + 512;
    ca->part_off = ca->sums_off + 8 * 2 * kClusterMaxTokens * 4;
    ca->sql_off = ca->part_off + part;
    ca->red_off = ca->sql_off + sql;
    ca->smem_bytes = ca->red_off + red + 1024;
    return ca->smem_bytes <= static_cast<uint32_t>(kClusterSmemMax);
}

mhc_status check_params(const mhc_params *p) {
    if (!p) return MHC_ERR_NULL;
    if (p->sinkhorn_iters < 1) return MHC_ERR_SHAPE;
    return MHC_OK;
}

CoefArgs coef_args(const float *scale, const float *base, const mhc_params *p) {
    CoefArgs c;
    c.scale = scale;
    c.base = base;
    c.hc_norm_eps = p->hc_norm_eps;
    c.hc_pre_eps = p->hc_pre_eps;
    c.hc_post_mult = p->hc_post_mult;
    c.sinkhorn_eps = p->sinkhorn_eps;
    c.norm_eps = p->norm_eps;
    c.sinkhorn_iters = p->sinkhorn_iters;
    return c;
}

mhc_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MHC_OK : MHC_ERR_CUDA; }

// Kernels this library has launched in the process (mhc_debug_launch_count).
std::atomic<unsigned long long> g_launches{0};
// The status of one kernel launch; counts it when it went out.
mhc_status launched(cudaError_t e) {
    if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
    return cuda_status(e);
}

// Shared body of mhc_pre (x == NULL) and mhc_boundary_fused.
mhc_status run_boundary(int mode, const uint16_t *x, const uint16_t *residual, const float *post,
                        const float *comb, const float *pre_lag, const void *weight,
                        const float *scale, const float *base, const void *norm_w,
                        mhc_dtype norm_dtype, const mhc_params *params, long long T, int H,
                        uint16_t *residual_out, uint16_t *layer_input, float *pre_out,
                        float *post_out, float *comb_out, void *workspace, size_t ws_bytes,
                        void *stream) {
    if (T < 0) return MHC_ERR_SHAPE;
    if (mhc_status s = check_params(params)) return s;
    if (!hidden_ok(H)) return MHC_ERR_UNSUPPORTED;
    if (norm_w && norm_dtype != MHC_F32 && norm_dtype != MHC_BF16) return MHC_ERR_SHAPE;
    if (T == 0) return MHC_OK;
    const bool fused = mode != PRE_ONLY;
    const void *need[] = {residual, weight, scale, base, layer_input, pre_out, post_out, comb_out,
                          workspace};
    for (const void *p : need)
        if (!p) return MHC_ERR_NULL;
    if (fused && (!x || !post || !comb || !residual_out)) return MHC_ERR_NULL;
    if (mode == FUSED_SHIFTED && !pre_lag) return MHC_ERR_NULL;
    const void *al[] = {x, residual, post, comb, pre_lag, weight, scale, base, norm_w,
                        residual_out, layer_input, pre_out, post_out, comb_out, workspace};
    for (const void *p : al)
        if (p && !aligned16(p)) return MHC_ERR_ALIGN;
    if (ws_bytes < workspace_bytes(T, H)) return MHC_ERR_WORKSPACE;

    const size_t nres = static_cast<size_t>(T) * 4 * H * 2, nx = static_cast<size_t>(T) * H * 2;
    const size_t n4 = static_cast<size_t>(T) * 16, n16 = static_cast<size_t>(T) * 64;
    const size_t nw = norm_w ? static_cast<size_t>(H) * (norm_dtype == MHC_BF16 ? 2 : 4) : 0;
    const Range ins[] = {{x, fused ? nx : 0}, {residual, nres}, {post, fused ? n4 : 0},
                         {comb, fused ? n16 : 0}, {pre_lag, pre_lag ? n4 : 0},
                         {weight, mhc_weight_bytes(H)}, {scale, 12}, {base, 96}, {norm_w, nw}};
    const Range outs[] = {{fused ? residual_out : nullptr, fused ? nres : 0},
                          {layer_input, nx}, {pre_out, n4}, {post_out, n4}, {comb_out, n16},
                          {workspace, ws_bytes}};
    if (aliasing(outs, 6, ins, 9, residual, residual_out)) return MHC_ERR_ALIAS;

    DeviceInfo *dev = nullptr;
    if (mhc_status s = current_device(&dev)) return s;
    if (!get_encoder()) return MHC_ERR_CUDA;

    const bool invariant = params->batch_invariant != 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *const ws8 = static_cast<uint8_t *>(workspace);
    const int path = g_decode_path.load();
    if (mode == FUSED_SHIFTED && !invariant && path != 1) {
        // a decode batch on one thread-block cluster: one kernel, no flags
        ClusterArgs ca;
        if (cluster_plan(T, H, &ca) && (path == 2 || cluster_preferred(T, ca)) &&
            cluster_fits(ca.ctas, ca.smem_bytes)) {
            CUtensorMap m_res, m_x, m_rout;
            if (!encode_cached(2, &m_res, residual, H, T) || !encode_cached(1, &m_x, x, H, T) ||
                !encode_cached(2, &m_rout, residual_out, H, T))
                return MHC_ERR_CUDA;
            ca.post = post;
            ca.comb = comb;
            ca.pre_lag = pre_lag;
            ca.weight = static_cast<const uint8_t *>(weight);
            ca.status = dev->status;
            ca.timeout_ns = g_timeout_ns.load();
            ca.coef = coef_args(scale, base, params);
            ca.norm_w = norm_w;
            ca.nw_bf16 = norm_dtype == MHC_BF16;
            ca.out32 = (reinterpret_cast<uintptr_t>(layer_input) & 31u) == 0;
            ca.layer_input = layer_input;
            ca.pre_out = pre_out;
            ca.post_out = post_out;
            ca.comb_out = comb_out;
            // the reduced mixes, after the epoch cell (the workspace holds
            // at least T x 128 bytes there for any plan)
            ca.mix_out = reinterpret_cast<float *>(ws8 + kCellBytes);
            ca.pdl = g_pdl.load();
            if (mhc_status s = launched(launch_cluster(m_res, m_x, m_rout, ca, st))) return s;
            if (t_between_event) {
                cudaEvent_t ev = t_between_event;
                t_between_event = nullptr;
                if (cudaEventRecord(ev, st) != cudaSuccess) return MHC_ERR_CUDA;
            }
            return MHC_OK;
        }
    }
    int S = 0, w = 0;
    if (invariant)
        plan_invariant(H, &S, &w);
    else
        plan(T, H, &S, &w);
    CUtensorMap m_res, m_x, m_rout;
    if (!encode_cached(0, &m_res, residual, H, T)) return MHC_ERR_CUDA;
    m_x = m_rout = m_res;
    if (fused) {
        if (!encode_cached(1, &m_x, x, H, T) || !encode_cached(0, &m_rout, residual_out, H, T))
            return MHC_ERR_CUDA;
    }
    StreamArgs sa;
    sa.post = post;
    sa.comb = comb;
    sa.pre_lag = pre_lag;
    sa.weight = static_cast<const uint8_t *>(weight);
    sa.partials = reinterpret_cast<float *>(ws8 + kCellBytes);
    sa.status = dev->status;
    sa.T = T;
    sa.H = H;
    sa.slice_w = w;
    sa.timeout_ns = g_timeout_ns.load();
    sa.ssql = reinterpret_cast<float *>(ws8 + kCellBytes + partials_bytes(T, S));
    sa.flags = reinterpret_cast<unsigned long long *>(ws8 + kCellBytes + partials_bytes(T, S) +
                                                      ssql_bytes(T, S));
    sa.epoch = 0;
    sa.epoch_cell = nullptr;
    sa.bump_cell = 0;
    sa.bump_poll = 0;
    sa.coef = coef_args(scale, base, params);
    sa.norm_w = norm_w;
    sa.nw_bf16 = norm_dtype == MHC_BF16;
    sa.out32 = (reinterpret_cast<uintptr_t>(layer_input) & 31u) == 0;
    sa.box_rows = box_rows_for(T);
    sa.pdl = g_pdl.load();
    sa.collapse_in_kernel = 0;
    sa.res_in = residual;
    sa.x_in = x;
    sa.layer_input = layer_input;
    sa.pre_out = pre_out;
    sa.post_out = post_out;
    sa.comb_out = comb_out;
    const long long tiles = (T + kTileT - 1) / kTileT;
    const long long items = tiles * S;
    if (items > 0x7FFFFFFFLL) return MHC_ERR_UNSUPPORTED;
    const int cap = dev->sms < kGridCap ? dev->sms : kGridCap;
    const int grid = static_cast<int>(items < cap ? items : cap);
    // the shifted form finishes in-kernel: every slice of a tile must be in
    // flight at once, and an item's collapse must fit its TMEM buffer
    if (mode == FUSED_SHIFTED && (S > grid || w / kChunk > 8)) return MHC_ERR_UNSUPPORTED;
    // the shifted form forms the coefficients in the streaming kernel, by
    // its workers: in a single wave of items as soon as the tile has
    // published (reduction split into ranges, for latency), otherwise after
    // the CTA's last item (reduction in slice order, as in the
    // batch-invariant plan). The unshifted forms do so for a single wave of
    // one tile whose CTAs own one round of tokens each (kRoundTok), and the
    // owner CTAs then write those tokens' layer input too
    // (collapse_in_kernel; else a collapse kernel follows): at 1 to 128
    // tokens and hidden 7168 forming them in-kernel took 0.4-2.4 us less
    // than the coefficients kernel between the two. With several rounds per
    // CTA the in-kernel reduction grows with them; those calls keep the
    // coefficients kernel.
    // (several tiles in one wave measured slower in-kernel: at 512 and 256
    // tokens, hidden 7168, 24.3 / 20.3 us unshifted with the coefficients in
    // the streaming kernel and a collapse kernel, 30.4 / 24.4 us with the
    // owners also writing the layer input, against 22.1 / 18.8 us with the
    // coefficients kernel between the two)
    const bool one_round = tiles == 1 && (T + S - 1) / S <= kRoundTok;
    sa.fuse_coef = items <= grid && !invariant && (mode == FUSED_SHIFTED || one_round);
    sa.coef_end = mode == FUSED_SHIFTED && !sa.fuse_coef;
    // the unshifted forms of a single wave write the layer input in the
    // streaming kernel too (the owner CTA recomputes each of its tokens'
    // updated residual from the inputs, so not when the update is in place)
    sa.collapse_in_kernel = mode != FUSED_SHIFTED && sa.fuse_coef && H <= kInKernelCollapseMaxH &&
                            !(mode == FUSED_UNSHIFTED && residual_out == residual);
    // the decode worker mapping (every worker warp on a quarter or half of
    // each hidden unit) for a single wave of one tile of at most 64 tokens
    // whose items fit the stages, in the fused forms (unshifted: 0.6-1.2 us
    // less at hidden 7168, 1 to 64 tokens)
    sa.decode_map = mode != PRE_ONLY && sa.fuse_coef && tiles == 1 && T <= kDecodeMaxTokens &&
                            w / kChunk <= kStreamStages
                        ? (T <= 32 ? 1 : 2)
                        : 0;
    if (sa.fuse_coef || mode == FUSED_SHIFTED) {
        // Flags hold a value unique to the call. A captured call replays with
        // its launch arguments frozen, so it takes the value from a cell in
        // the workspace (plus one) and advances the cell itself once every
        // CTA has read it: CTA 0 does, after it has seen every CTA publish
        // (a call of one tile in a single wave, whose CTA 0 waits for them
        // all anyway) or every CTA's first item publish (any other call).
        // Calls outside a capture get the value from the host.
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return MHC_ERR_CUDA;
        if (cap == cudaStreamCaptureStatusActive) {
            sa.epoch_cell = reinterpret_cast<unsigned long long *>(ws8);
            sa.bump_cell = sa.fuse_coef && tiles == 1;
            sa.bump_poll = !sa.bump_cell;
        } else {
            sa.epoch = next_epoch();
        }
    }
    if (mhc_status s = launched(launch_stream(mode, m_res, m_x, m_rout, sa, S,
                                                 static_cast<int>(items), grid, st)))
        return s;
    if (t_between_event) {
        cudaEvent_t ev = t_between_event;
        t_between_event = nullptr;
        if (cudaEventRecord(ev, st) != cudaSuccess) return MHC_ERR_CUDA;
    }

    FinishArgs fa;
    fa.partials = reinterpret_cast<const float *>(ws8 + kCellBytes);
    fa.n_slices = S;
    fa.coef = coef_args(scale, base, params);
    fa.norm_w = norm_w;
    fa.nw_bf16 = norm_dtype == MHC_BF16;
    fa.cur = mode == FUSED_UNSHIFTED ? residual_out : residual;
    fa.layer_input = layer_input;
    fa.pre_out = pre_out;
    fa.post_out = post_out;
    fa.comb_out = comb_out;
    fa.T = T;
    fa.H = H;
    if (mode == FUSED_SHIFTED || sa.collapse_in_kernel) return MHC_OK;
    if (!sa.fuse_coef)
        if (mhc_status s = launched(launch_coefficients(fa, st))) return s;
    // after the coefficients kernel, as its programmatic dependent (released
    // once every block has written its coefficients) for pre-only calls of up
    // to 2048 tokens and unshifted ones of up to 512: at hidden 7168 1.2-2.2
    // us less per pre-only call from 512 to 2048 tokens and 2.5 us less per
    // unshifted call at 512, but 0.3-0.7 us more per unshifted call at 1024
    // and 2048, and 4-12 us more per call at 8192. Directly after the
    // streaming kernel (which releases its dependents at its start) a plain
    // launch.
    const bool pdl_collapse = !sa.fuse_coef && T <= (mode == PRE_ONLY ? 2048 : 512);
    // (batch-invariant calls keep one block size, so that the collapse's sum
    // of squares has one order at every batch size)
    return launched(launch_collapse_unshifted(fa, st, pdl_collapse, !invariant && T <= dev->sms));
}

}  // namespace

extern "C" {

size_t mhc_weight_bytes(int hidden) {
    return hidden_ok(hidden) ? static_cast<size_t>(384) * hidden : 0;
}

size_t mhc_workspace_bytes(int64_t tokens, int hidden) { return workspace_bytes(tokens, hidden); }

mhc_status mhc_plan(int64_t tokens, int hidden, int *n_slices, int *slice_width) {
    if (!n_slices || !slice_width) return MHC_ERR_NULL;
    if (tokens < 0) return MHC_ERR_SHAPE;
    if (!hidden_ok(hidden)) return MHC_ERR_UNSUPPORTED;
    plan(tokens, hidden, n_slices, slice_width);
    return MHC_OK;
}

mhc_status mhc_prepare_weight(const float *fn, int hidden, void *weight, void *stream) {
    if (!hidden_ok(hidden)) return MHC_ERR_UNSUPPORTED;
    if (!fn || !weight) return MHC_ERR_NULL;
    if (!aligned16(fn) || !aligned16(weight)) return MHC_ERR_ALIGN;
    if (overlap(fn, static_cast<size_t>(96) * 4 * hidden, weight, mhc_weight_bytes(hidden)))
        return MHC_ERR_ALIAS;
    DeviceInfo *dev = nullptr;
    if (mhc_status s = current_device(&dev)) return s;
    return launched(launch_prepare_weight(fn, hidden, static_cast<uint8_t *>(weight),
                                             static_cast<cudaStream_t>(stream)));
}

mhc_status mhc_post(const uint16_t *x, const uint16_t *residual, const float *post,
                    const float *comb, uint16_t *residual_out, int64_t tokens, int hidden,
                    void *stream) {
    if (tokens < 0) return MHC_ERR_SHAPE;
    if (!hidden_ok(hidden)) return MHC_ERR_UNSUPPORTED;
    if (tokens == 0) return MHC_OK;
    if (!x || !residual || !post || !comb || !residual_out) return MHC_ERR_NULL;
    const void *al[] = {x, residual, post, comb, residual_out};
    for (const void *p : al)
        if (!aligned16(p)) return MHC_ERR_ALIGN;
    const size_t nres = static_cast<size_t>(tokens) * 4 * hidden * 2;
    const Range ins[] = {{x, static_cast<size_t>(tokens) * hidden * 2}, {residual, nres},
                         {post, static_cast<size_t>(tokens) * 16},
                         {comb, static_cast<size_t>(tokens) * 64}};
    const Range outs[] = {{residual_out, nres}};
    if (aliasing(outs, 1, ins, 4, residual, residual_out)) return MHC_ERR_ALIAS;
    DeviceInfo *dev = nullptr;
    if (mhc_status s = current_device(&dev)) return s;
    return launched(launch_post(x, residual, post, comb, residual_out, tokens, hidden,
                                   static_cast<cudaStream_t>(stream)));
}

mhc_status mhc_pre(const uint16_t *residual, const void *weight, const float *scale,
                   const float *base, const void *norm_w, mhc_dtype norm_dtype,
                   const mhc_params *params, int64_t tokens, int hidden, uint16_t *layer_input,
                   float *pre_out, float *post_out, float *comb_out, void *workspace,
                   size_t workspace_bytes, void *stream) {
    return run_boundary(PRE_ONLY, nullptr, residual, nullptr, nullptr, nullptr, weight, scale,
                        base, norm_w, norm_dtype, params, tokens, hidden, nullptr, layer_input,
                        pre_out, post_out, comb_out, workspace, workspace_bytes, stream);
}

mhc_status mhc_pre_split_k(const uint16_t *residual, const float *dot_mix, const float *sqrsum,
                           int n_splits, const float *scale, const float *base,
                           const void *norm_w, mhc_dtype norm_dtype, const mhc_params *params,
                           int64_t tokens, int hidden, uint16_t *layer_input, float *pre_out,
                           float *post_out, float *comb_out, void *stream) {
    const long long T = tokens;
    const int H = hidden;
    if (T < 0 || n_splits < 1 || n_splits > kMaxSplits) return MHC_ERR_SHAPE;
    if (mhc_status s = check_params(params)) return s;
    if (!hidden_ok(H)) return MHC_ERR_UNSUPPORTED;
    if (norm_w && norm_dtype != MHC_F32 && norm_dtype != MHC_BF16) return MHC_ERR_SHAPE;
    if (T == 0) return MHC_OK;
    const void *need[] = {residual, dot_mix, sqrsum, scale, base, layer_input, pre_out, post_out,
                          comb_out};
    for (const void *p : need)
        if (!p) return MHC_ERR_NULL;
    const void *al[] = {residual, dot_mix, sqrsum, scale, base, norm_w, layer_input, pre_out,
                        post_out, comb_out};
    for (const void *p : al)
        if (p && !aligned16(p)) return MHC_ERR_ALIGN;
    const size_t nres = static_cast<size_t>(T) * 4 * H * 2, nx = static_cast<size_t>(T) * H * 2;
    const size_t n4 = static_cast<size_t>(T) * 16, n16 = static_cast<size_t>(T) * 64;
    const size_t nmix = static_cast<size_t>(n_splits) * T * 24 * 4;
    const size_t nsq = static_cast<size_t>(n_splits) * T * 4;
    const size_t nw = norm_w ? static_cast<size_t>(H) * (norm_dtype == MHC_BF16 ? 2 : 4) : 0;
    const Range ins[] = {{residual, nres}, {dot_mix, nmix}, {sqrsum, nsq}, {scale, 12},
                         {base, 96}, {norm_w, nw}};
    const Range outs[] = {{layer_input, nx}, {pre_out, n4}, {post_out, n4}, {comb_out, n16}};
    if (aliasing(outs, 4, ins, 6, nullptr, nullptr)) return MHC_ERR_ALIAS;
    DeviceInfo *dev = nullptr;
    if (mhc_status s = current_device(&dev)) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    FinishArgs fa;
    fa.partials = nullptr;
    fa.n_slices = 0;
    fa.coef = coef_args(scale, base, params);
    fa.norm_w = norm_w;
    fa.nw_bf16 = norm_dtype == MHC_BF16;
    fa.cur = residual;
    fa.layer_input = layer_input;
    fa.pre_out = pre_out;
    fa.post_out = post_out;
    fa.comb_out = comb_out;
    fa.T = T;
    fa.H = H;
    // few tokens: one kernel, the collapse overlapping the coefficients
    // (latency); many: coefficients for 32 tokens per block, then the
    // collapse (bandwidth)
    if (T <= kSplitKOneKernelTokens && !params->batch_invariant)
        return launched(launch_pre_split_k(dot_mix, sqrsum, n_splits, fa, st, T <= dev->sms));
    if (mhc_status s = launched(launch_coefficients_split_k(dot_mix, sqrsum, n_splits, fa, st)))
        return s;
    // as a programmatic dependent of the coefficients kernel (released after
    // its coefficients): 0.66 us less at 1536 x 4096, 0.35 at 2048 x 7168,
    // unchanged at 4096 tokens
    return launched(launch_collapse_unshifted(fa, st, true, !params->batch_invariant && T <= dev->sms));
}

mhc_status mhc_boundary_fused(const uint16_t *x, const uint16_t *residual, const float *post,
                              const float *comb, const float *pre_lag, const void *weight,
                              const float *scale, const float *base, const void *norm_w,
                              mhc_dtype norm_dtype, const mhc_params *params, int64_t tokens,
                              int hidden, uint16_t *residual_out, uint16_t *layer_input,
                              float *pre_out, float *post_out, float *comb_out, void *workspace,
                              size_t workspace_bytes, void *stream) {
    return run_boundary(pre_lag ? FUSED_SHIFTED : FUSED_UNSHIFTED, x, residual, post, comb,
                        pre_lag, weight, scale, base, norm_w, norm_dtype, params, tokens, hidden,
                        residual_out, layer_input, pre_out, post_out, comb_out, workspace,
                        workspace_bytes, stream);
}

mhc_status mhc_plan_cluster(int64_t tokens, int hidden, int *ctas) {
    if (!ctas) return MHC_ERR_NULL;
    *ctas = 0;
    if (tokens < 0) return MHC_ERR_SHAPE;
    if (!hidden_ok(hidden)) return MHC_ERR_UNSUPPORTED;
    DeviceInfo *dev = nullptr;
    if (mhc_status s = current_device(&dev)) return s;
    ClusterArgs ca;
    const int path = g_decode_path.load();
    if (path != 1 && cluster_plan(tokens, hidden, &ca) &&
        (path == 2 || cluster_preferred(tokens, ca)) && cluster_fits(ca.ctas, ca.smem_bytes))
        *ctas = ca.ctas;
    return MHC_OK;
}

void mhc_debug_set_pdl(int enable) { g_pdl.store(enable ? 1 : 0); }

uint64_t mhc_debug_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

mhc_status mhc_debug_delayed_copy(const uint16_t *src, uint16_t *dst, int64_t n,
                                  uint32_t delay_ns, void *stream) {
    if (n < 0 || delay_ns > 1000000u) return MHC_ERR_SHAPE;
    if (n == 0) return MHC_OK;
    if (!src || !dst) return MHC_ERR_NULL;
    if (!aligned16(src) || !aligned16(dst)) return MHC_ERR_ALIGN;
    if (overlap(src, static_cast<size_t>(n) * 2, dst, static_cast<size_t>(n) * 2)) return MHC_ERR_ALIAS;
    DeviceInfo *dev = nullptr;
    if (mhc_status s = current_device(&dev)) return s;
    return launched(launch_delayed_copy(src, dst, n, delay_ns, static_cast<cudaStream_t>(stream)));
}

void mhc_debug_set_decode_path(int path) { g_decode_path.store(path == 1 || path == 2 ? path : 0); }

mhc_status mhc_get_device_status(void *stream) {
    DeviceInfo *dev = nullptr;
    if (mhc_status s = current_device(&dev)) return s;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MHC_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpy(&word, dev->status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return MHC_ERR_CUDA;
    if (word == 0) return MHC_OK;
    if (cudaMemset(dev->status, 0, sizeof word) != cudaSuccess) return MHC_ERR_CUDA;
    t_last_site = static_cast<int>(word >> 8);
    const int code = static_cast<int>(word & 0xFF);
    return code == MHC_ERR_DEVICE_TIMEOUT ? MHC_ERR_DEVICE_TIMEOUT : MHC_ERR_CUDA;
}

int mhc_last_timeout_site(void) { return t_last_site; }

const char *mhc_status_string(mhc_status s) {
    switch (s) {
        case MHC_OK: return "MHC_OK";
        case MHC_ERR_NULL: return "MHC_ERR_NULL: a required pointer is NULL";
        case MHC_ERR_ALIGN: return "MHC_ERR_ALIGN: a pointer is not 16-byte aligned";
        case MHC_ERR_SHAPE: return "MHC_ERR_SHAPE: bad token count or parameters";
        case MHC_ERR_UNSUPPORTED: return "MHC_ERR_UNSUPPORTED: hidden size or device not supported";
        case MHC_ERR_ALIAS: return "MHC_ERR_ALIAS: an output overlaps an input or another output";
        case MHC_ERR_CUDA: return "MHC_ERR_CUDA: a CUDA call failed";
        case MHC_ERR_DEVICE_TIMEOUT: return "MHC_ERR_DEVICE_TIMEOUT: a device-side wait ran out";
        case MHC_ERR_WORKSPACE: return "MHC_ERR_WORKSPACE: workspace missing or too small";
    }
    return "unknown mhc_status";
}

void mhc_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : 1000000000ull); }

void mhc_debug_record_between(void *event) {
    t_between_event = static_cast<cudaEvent_t>(event);
}

mhc_status mhc_debug_unarmed_wait(void *stream) {
    DeviceInfo *dev = nullptr;
    if (mhc_status s = current_device(&dev)) return s;
    return launched(
        launch_unarmed_wait(dev->status, g_timeout_ns.load(), static_cast<cudaStream_t>(stream)));
}

mhc_status mhc_debug_coef_check(const float *values, const float *scale, const float *base,
                                const mhc_params *params, int hidden, int64_t tokens,
                                float *out_thread, float *out_lanes, void *stream) {
    if (tokens < 0) return MHC_ERR_SHAPE;
    if (mhc_status s = check_params(params)) return s;
    if (!hidden_ok(hidden)) return MHC_ERR_UNSUPPORTED;
    if (tokens == 0) return MHC_OK;
    const void *need[] = {values, scale, base, out_thread, out_lanes};
    for (const void *p : need) {
        if (!p) return MHC_ERR_NULL;
        if (!aligned16(p)) return MHC_ERR_ALIGN;
    }
    if (tokens > 0x7FFFFFFFLL * 32) return MHC_ERR_SHAPE;
    const size_t nv = static_cast<size_t>(tokens) * 25 * 4, no = static_cast<size_t>(tokens) * 24 * 4;
    const Range ins[] = {{values, nv}, {scale, 12}, {base, 96}};
    const Range outs[] = {{out_thread, no}, {out_lanes, no}};
    if (aliasing(outs, 2, ins, 3, nullptr, nullptr)) return MHC_ERR_ALIAS;
    DeviceInfo *dev = nullptr;
    if (mhc_status s = current_device(&dev)) return s;
    return launched(launch_coef_check(values, coef_args(scale, base, params), hidden, tokens,
                                         out_thread, out_lanes, static_cast<cudaStream_t>(stream)));
}

mhc_status mhc_debug_rcp_check(uint32_t first_bits, uint64_t count, unsigned long long *result,
                               void *stream) {
    if (!result) return MHC_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(result) & 7u) != 0) return MHC_ERR_ALIGN;
    if (count == 0) return MHC_OK;
    if (count > (1ull << 32) - first_bits) return MHC_ERR_SHAPE;
    DeviceInfo *dev = nullptr;
    if (mhc_status s = current_device(&dev)) return s;
    return launched(launch_rcp_check(first_bits, count, result,
                                        static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
