// Internal declarations shared by the kernel translation units and the host
// API. Not part of the C ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mhc {

enum Mode : int { PRE_ONLY = 0, FUSED_UNSHIFTED = 1, FUSED_SHIFTED = 2 };

constexpr int kTileT = 128;                         // tokens per CTA tile (MMA M)
constexpr int kChunk = 32;                          // hidden per pipeline stage
constexpr int kRowBytes = kChunk * 2;               // one 64-byte bf16 row
constexpr int kResBytes = 4 * kTileT * kRowBytes;   // residual / cur tile
constexpr int kXBytes = kTileT * kRowBytes;         // x / collapse tile
constexpr int kWRows = 48;                          // 24 hi + 24 lo weight rows
constexpr int kWBytes = 4 * kWRows * kRowBytes;     // weight tile of one chunk
constexpr int kStageBytes = kResBytes + kXBytes + kWBytes;
// Partials of one (tile, slice) item, a block of kItemFloats fp32: per token,
// values 0-23 the partial mixes (hi + lo), 24 the partial 4H sum of squares.
// Value-major [kPartVals][kTileT] (a warp reads or writes one value of 32
// tokens as one 128-byte row) in general; token-major [kTileT][kTokStride]
// (16-byte aligned runs) when the call is a single wave of items and the
// shifted streaming kernel's workers reduce them for a few tokens each.
// Multi-item shifted calls use a third layout: per token a 32-float record
// for each slice, [T rounded up to tiles][S][kRecFloats] (a 4-token group's
// records of every slice are one contiguous run, fetched by one bulk copy).
constexpr int kPartVals = 25;
constexpr int kTokStride = 28;
constexpr int kRecFloats = 32;
constexpr int kItemFloats = kTileT * kRecFloats;    // one item's share of the workspace

struct CoefArgs {
    const float *scale;
    const float *base;
    float hc_norm_eps, hc_pre_eps, hc_post_mult, sinkhorn_eps, norm_eps;
    int sinkhorn_iters;
};

struct StreamArgs {
    const float *post;       // [T,4]
    const float *comb;       // [T,4,4]
    const float *pre_lag;    // [T,4] (shifted only)
    const uint8_t *weight;   // prepared tiles
    float *partials;         // [tiles][n_slices] item blocks of kItemFloats
    unsigned int *status;    // device status word
    long long T;
    int H;
    int slice_w;             // hidden per slice (multiple of kChunk)
    unsigned long long timeout_ns;
    // shifted form: the kernel also finishes the boundary
    float *ssql;                 // [n_slices][T] per-slice sums of the collapse's squares
    unsigned long long *flags;   // [tiles][n_slices][4] per-call epoch flags
    unsigned long long epoch;    // this call's flag value (epoch_cell == NULL)
    unsigned long long *epoch_cell;   // else: the flag value is the cell's plus one,
                                      // and the call advances the cell itself:
    int bump_cell;               // one tile: CTA 0's finishers, once they have seen
                                 // every CTA publish
    int bump_poll;               // several tiles: warp 2 of CTA 0, once every CTA's
                                 // first item has published
    CoefArgs coef;
    const void *norm_w;          // [H] or NULL
    int nw_bf16;
    int out32;                   // layer_input 32-byte aligned
    uint16_t *layer_input;       // [T,H]
    float *pre_out, *post_out, *comb_out;
    int fuse_coef;               // one item per CTA: the workers form the coefficients
    int coef_end;                // shifted, several items per CTA: the workers form
                                 // them after the CTA's last item (record layout)
    int decode_map;              // one tile of at most kDecodeMaxTokens tokens in a single
                                 // wave, at most kStreamStages chunks, fused forms: the decode
                                 // mapping of the worker warps, 1 up to 32 tokens, 2 above
                                 // (shifted: the collapse kept in the stage's x tile; see the
                                 // streaming kernel); 0 otherwise
    int box_rows;                // one tile: token rows per residual / x box (the
                                 // residual maps then hold one stream per box); 0: 128
    int pdl;                     // launch as a programmatic dependent of the previous kernel
    // unshifted forms, single wave (fuse_coef), H <= kInKernelCollapseMaxH and not in place:
    // each owner CTA also writes its tokens' layer input (no collapse kernel after it),
    // recomputing the token's updated residual from the inputs
    int collapse_in_kernel;
    const uint16_t *res_in;      // [T,4,H] the residual input
    const uint16_t *x_in;        // [T,H] the layer output (fused form)
};

// Largest hidden size whose unshifted single-wave calls collapse in the
// streaming kernel (each of the owner CTA's 256 worker threads keeps up to
// 4 units of 8 collapse values of the token in registers).
constexpr int kInKernelCollapseMaxH = 8 * 256 * 4;

struct FinishArgs {
    const float *partials;   // [tiles][n_slices] value-major item blocks of kItemFloats
    int n_slices;
    CoefArgs coef;
    const void *norm_w;      // [H] or NULL
    int nw_bf16;
    const uint16_t *cur;     // [T,4,H] stream the collapse reads (unshifted)
    uint16_t *layer_input;   // [T,H]
    float *pre_out, *post_out, *comb_out;   // the collapse reads pre_out
    long long T;
    int H;
};

// Decode calls on one thread-block cluster: at most this many tokens (one
// tile, a quarter of the worker warps' lanes per token at most), at most
// kClusterMaxCtas CTAs (hidden slices), each with at most kClusterMaxChunks
// chunks of 32 and kClusterMaxStages pipeline stages.
constexpr int kClusterMaxTokens = 64;
constexpr int kClusterMaxCtas = 16;
constexpr int kClusterMaxChunks = 32;
constexpr int kClusterMaxStages = 16;
constexpr int kClusterRecFloats = 28;               // a token's 25 values pushed to its owner, padded
constexpr int kClusterSmemMax = 232448;             // dynamic shared memory per CTA (227 KB)

// Arguments of the cluster kernel: one cluster of `ctas` CTAs, CTA r owning
// hidden chunks r, r + ctas, ... (nch of them) of the one tile of T tokens.
// Shared-memory offsets are from the 1024-byte-aligned base.
struct ClusterArgs {
    const float *post;       // [T,4]
    const float *comb;       // [T,4,4]
    const float *pre_lag;    // [T,4]
    const uint8_t *weight;   // prepared tiles
    unsigned int *status;    // device status word
    unsigned long long timeout_ns;
    int T, H;
    int ctas;                // cluster size = hidden slices
    int nch;                 // chunks per CTA
    int rows;                // token rows per box (T rounded up to 8)
    int stages;              // pipeline stages (== nch when every chunk stays resident)
    uint32_t stage_bytes;    // 4 residual boxes + the x box + a 12 KB weight tile
    uint32_t li_off;         // the CTA's collapse [nch][rows][32] bf16 (unswizzled)
    uint32_t bar_off;        // mbarriers and the TMEM slot / abort flag
    uint32_t sums_off;       // worker warps' per-token sums [8][2][64] fp32
    uint32_t part_off;       // owned tokens' pushed values [owned][ctas][kClusterRecFloats]
    uint32_t sql_off;        // every CTA's collapse sums of squares [ctas][T] fp32
    uint32_t red_off;        // coefficient reduction [16][25], constants [32], rstd_li [64]
    uint32_t smem_bytes;     // dynamic shared memory of the launch
    CoefArgs coef;
    const void *norm_w;      // [H] or NULL
    int nw_bf16;
    int out32;               // layer_input 32-byte aligned
    uint16_t *layer_input;   // [T,H]
    float *pre_out, *post_out, *comb_out;
    float *mix_out;          // [T][kClusterRecFloats]: each token's reduced 24 mixes and
                             // 4H sum of squares, kept in the caller's scratch (or NULL)
    int pdl;                 // launch as a programmatic dependent of the previous kernel
};

constexpr int kGridCap = 152;                       // persistent CTAs: one per GB300 SM
constexpr int kStreamStages = 4;                    // pipeline stages of the streaming kernel
constexpr int kDecodeMaxTokens = 64;                // most tokens of the decode worker mapping
constexpr int kRoundTok = 5;                        // single wave: tokens per coefficient round
constexpr int kMaxSplits = 64;                      // split-K pre: most K splits accepted

size_t stream_smem_bytes();
// Persistent streaming kernel over n_items = tiles x n_slices work items
// (item i = tile i / n_slices, slice i % n_slices), `grid` CTAs.
cudaError_t launch_stream(int mode, const CUtensorMap &res, const CUtensorMap &x,
                          const CUtensorMap &rout, const StreamArgs &a, int n_slices, int n_items,
                          int grid, cudaStream_t s);
// Shifted decode call on one thread-block cluster of a.ctas CTAs (the hidden
// slices exchange their partials through distributed shared memory).
cudaError_t launch_cluster(const CUtensorMap &res, const CUtensorMap &x, const CUtensorMap &rout,
                           const ClusterArgs &a, cudaStream_t s);
// Whether a cluster of `ctas` CTAs with `smem` bytes of dynamic shared memory
// can be resident on the current device (checked once per size and device).
bool cluster_fits(int ctas, uint32_t smem);
// pdl: as a programmatic dependent of the kernel before it (which must
// release it only once the pre it reads is written)
// wide: 512 threads per token (every token on an SM of its own), else 128
cudaError_t launch_collapse_unshifted(const FinishArgs &a, cudaStream_t s, bool pdl, bool wide);
cudaError_t launch_coefficients(const FinishArgs &a, cudaStream_t s);
// wide: 512 threads per token (every token on an SM of its own), else 128
cudaError_t launch_pre_split_k(const float *dot_mix, const float *sqrsum, int n_splits,
                               const FinishArgs &a, cudaStream_t s, bool wide);
cudaError_t launch_coefficients_split_k(const float *dot_mix, const float *sqrsum, int n_splits,
                                        const FinishArgs &a, cudaStream_t s);
cudaError_t launch_prepare_weight(const float *fn, int H, uint8_t *out, cudaStream_t s);
cudaError_t launch_post(const uint16_t *x, const uint16_t *res, const float *post,
                        const float *comb, uint16_t *out, long long T, int H, cudaStream_t s);
cudaError_t launch_unarmed_wait(unsigned int *status, unsigned long long timeout_ns,
                                cudaStream_t s);
// Advances the u64 at `cell` by one (a single thread): the flag value of the
// shifted call that follows on the stream, when that call is being captured.
cudaError_t launch_coef_check(const float *v, const CoefArgs &c, int H, long long n,
                              float *out_thread, float *out_lanes, cudaStream_t s);
// Test producer: lets the next kernel on the stream start at once, waits
// delay_ns (bounded), then copies n bf16 values src -> dst.
cudaError_t launch_delayed_copy(const uint16_t *src, uint16_t *dst, long long n, uint32_t delay_ns,
                                cudaStream_t s);
cudaError_t launch_rcp_check(uint32_t first, unsigned long long count, unsigned long long *out,
                             cudaStream_t s);
unsigned int *device_status_word();   // of the current device; NULL on failure

}  // namespace mhc
