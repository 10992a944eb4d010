/*
 * mhc.h: C ABI of the GB300 (sm_103a) mHC layer boundary, n_hc = 4.
 *
 * The boundary between layer l and l+1 of a manifold-constrained
 * hyper-connection stack, per token (X_{l+1} = B_l X_l + C_l F_l(A_l X_l),
 * "The Hyper Connection Preprocessing GPU Kernel Study", section "why this
 * kernel is called pre"):
 *   post  (residual update): residual'[s] = bf16(post[s]*x + sum_j comb[j][s]*residual[j])
 *   pre   (coefficients and layer input of the next layer): sum of squares of
 *         the flattened 4H residual -> rstd; 24 mixes = TF32(fn) . residual;
 *         pre = sigmoid(..)+eps, post = 2 sigmoid(..), comb = Sinkhorn(softmax(..));
 *         layer_input = bf16(bf16(sum_j pre[j]*residual[j]) * rstd_li * norm_w).
 * The fused entry point does both in one pass over the residual; its shifted
 * form collapses with the previous boundary's pre ("vllm.models.deepseek_v41
 * .nvidia.ops.mhc_boundary", mhc_shifted_post_pre_boundary).
 *
 * Conventions for every entry point below.
 *   - Tensors are plain, contiguous, row-major buffers. "bf16" buffers hold
 *     bfloat16 bit patterns as uint16_t. Unless stated otherwise a pointer is a
 *     DEVICE pointer on the current CUDA device, owned by the caller; the
 *     library never frees or retains it past the call.
 *   - Every pointer must be 16-byte aligned (MHC_ERR_ALIGN otherwise).
 *   - tokens T >= 0 (T == 0 is a no-op returning MHC_OK); hidden H must be a
 *     multiple of 32 in [32, 65536] (MHC_ERR_UNSUPPORTED otherwise).
 *   - stream is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Work is enqueued asynchronously; argument errors are returned before
 *     anything is enqueued. A launch failure returns MHC_ERR_CUDA.
 *   - No entry point allocates device memory. Scratch space, where needed, is
 *     the caller's `workspace` (see mhc_workspace_bytes).
 *   - Device-side waits are bounded: a kernel whose wait runs out records
 *     MHC_ERR_DEVICE_TIMEOUT in a per-device status word and returns early;
 *     read it with mhc_get_device_status().
 *   - Outputs must not overlap inputs or each other, except that
 *     residual_out may be exactly the residual buffer (in-place update).
 *     Partial overlap returns MHC_ERR_ALIAS.
 *   - Entry points are thread-safe; results are deterministic run to run
 *     for a given (T, H) (fixed reduction order).
 */
#ifndef MHC_H
#define MHC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MHC_OK = 0,
    MHC_ERR_NULL = 1,           /* a required pointer is NULL */
    MHC_ERR_ALIGN = 2,          /* a pointer is not 16-byte aligned */
    MHC_ERR_SHAPE = 3,          /* negative T, bad params (sinkhorn_iters < 1) */
    MHC_ERR_UNSUPPORTED = 4,    /* H outside the supported set, or not an sm_103 device */
    MHC_ERR_ALIAS = 5,          /* an output overlaps an input or another output */
    MHC_ERR_CUDA = 6,           /* a CUDA runtime/driver call failed */
    MHC_ERR_DEVICE_TIMEOUT = 7, /* a device-side bounded wait ran out */
    MHC_ERR_WORKSPACE = 8       /* workspace NULL or smaller than mhc_workspace_bytes */
} mhc_status;

/* Scalar parameters of a boundary ("mhc_boundary" page, mhc_shifted_post_pre_boundary
 * arguments hc_norm_eps, hc_pre_eps, hc_post_scale, sinkhorn_eps,
 * num_sinkhorn_iters, norm_eps). */
typedef struct {
    float hc_norm_eps;   /* eps inside rstd = rsqrt(ssq / (4H) + hc_norm_eps) */
    float hc_pre_eps;    /* pre = sigmoid(.) + hc_pre_eps */
    float hc_post_mult;  /* post = sigmoid(.) * hc_post_mult (2 in DeepSeek) */
    float sinkhorn_eps;  /* softmax floor and Sinkhorn denominator eps */
    float norm_eps;      /* eps of the layer RMSNorm of the collapse (over H) */
    int sinkhorn_iters;  /* >= 1: one column step, then iters-1 (row, column) steps */
    int batch_invariant; /* nonzero: every output of a token is bitwise the same
                          * whatever the batch it comes in (its size, its
                          * position): the hidden-slice plan then depends on
                          * the hidden size only and every reduction runs in
                          * one fixed order. The pages have no counterpart.
                          * Costs latency on small batches (fewer slices). */
} mhc_params;

/* Element type of norm_w. The DeepSeek boundary kernel reads bf16 weights;
 * fp32 is the common checkpoint dtype. */
typedef enum { MHC_F32 = 0, MHC_BF16 = 1 } mhc_dtype;

/* ---------------------------------------------------------------------- */
/* Weight preparation ("mhc_boundary" page, prepare_boundary_weight).       */

/* Bytes of the prepared mixer for hidden H: 48 rows x 4H bf16 = 384*H. */
size_t mhc_weight_bytes(int hidden);

/*
 * fn: [24, 4H] fp32, rows 0-3 pre, 4-7 post, 8-23 comb (row-major 4x4),
 *     column s*H + h multiplies stream s, hidden h of the residual.
 * weight: output, mhc_weight_bytes(H) bytes, 16-byte aligned.
 *
 * Each weight w is rounded to TF32 (round half away from zero on the bit
 * pattern: r = (bits(w) + 0x1000) & ~0x1FFF) and split into two bf16 parts,
 * hi = bf16_rne(r) and lo = bf16_rne(r - hi), with hi + lo == r exactly, so
 * BF16 tensor-core products reproduce TF32 products exactly. Layout (uint16
 * units): stacked row r in [0, 48) holds hi of mix r (r < 24) or lo of mix
 * r - 24; for hidden chunk c in [0, H/32), stream s and element e in [0, 32)
 * the value for column k = s*H + 32c + e is at
 *     ((c*4 + s)*48 + r)*32 + 8*((e/8) ^ ((r/2) % 4)) + (e % 8),
 * i.e. per (chunk, stream) a 48 x 64-byte tile, K-major, in the 64-byte
 * swizzled order the tensor cores read from shared memory.
 * This layout deliberately departs from the page's prepared weight, which
 * gathers the same hi/lo parts into register fragments of the warp-level
 * m16n8k16 MMA ([16 slices, k16 steps, 3 m16 tiles, 32 lanes, 4] int32):
 * here the 5th-generation tensor cores read both operands from shared
 * memory, so each (chunk, stream) tile lands there with one bulk copy,
 * already in the swizzled order their descriptors expect. The rounding and
 * the split are the page's, value for value.
 * Inputs must be finite (NaN payloads are not preserved by the rounding).
 */
mhc_status mhc_prepare_weight(const float *fn, int hidden, void *weight, void *stream);

/* ---------------------------------------------------------------------- */
/* Residual update alone ("mhc_boundary" page, residual_update).            */

/*
 * x: [T, H] bf16 layer output; residual: [T, 4, H] bf16; post: [T, 4] fp32;
 * comb: [T, 4, 4] fp32 where comb[t][j][s] carries stream j into stream s.
 * residual_out: [T, 4, H] bf16 (may be == residual).
 *   residual_out[t][s][h] = bf16_rne(chain), chain = post[s]*x[h], then
 *   fma(comb[j][s], residual[j][h], chain) for j = 0..3, every operand and
 *   result of the chain flushed to zero when subnormal.
 */
mhc_status mhc_post(const uint16_t *x, const uint16_t *residual, const float *post,
                    const float *comb, uint16_t *residual_out, int64_t tokens,
                    int hidden, void *stream);

/* ---------------------------------------------------------------------- */
/* Pre and fused boundary.                                                  */

/* Bytes of caller-provided device scratch for mhc_pre / mhc_boundary_fused
 * at (T, H): per-token partial mixes and sums of squares of every hidden
 * slice, and the publication flags. 0 when T == 0. It needs no
 * initialisation. Calls may be captured into a CUDA graph (they allocate
 * nothing and never synchronise). A call whose blocks wait on one another
 * (every shifted call, and the unshifted calls of at most 128 tokens whose
 * streaming kernel forms the coefficients) marks its progress with a flag
 * value; captured, it takes the value from a cell in the workspace and
 * advances the cell itself, so each replay has its own value and replays
 * may run with new contents in the same buffers (no extra kernel). Calls
 * that share a workspace must not overlap in time. The cell sits at the
 * start of the workspace whatever the call's shape, so calls of different
 * shapes, eager or captured, may share one workspace sized for the largest. */
size_t mhc_workspace_bytes(int64_t tokens, int hidden);

/*
 * Unshifted pre ("The Hyper Connection Preprocessing GPU Kernel Study",
 * mhc_pre_big_fuse with the in-kernel square sum; mixes computed in-kernel).
 * residual: [T, 4, H] bf16. weight: from mhc_prepare_weight(fn, H).
 * scale: [3] fp32 (pre, post, comb). base: [24] fp32 (rows of fn).
 * norm_w: [H] of norm_dtype, or NULL to write the raw collapse.
 * Outputs: layer_input [T, H] bf16, pre_out [T, 4], post_out [T, 4],
 * comb_out [T, 4, 4] fp32.
 *   ssq = sum over the 4H values of residual^2, rstd = rsqrt(ssq/(4H) + hc_norm_eps)
 *   mix[n] = sum_k TF32(fn[n][k]) * residual_flat[k]        (fp32 accumulate)
 *   pre[i] = sigmoid(fma(mix[i]*rstd, scale[0], base[i])) + hc_pre_eps
 *   post[i] = sigmoid(fma(mix[4+i]*rstd, scale[1], base[4+i])) * hc_post_mult
 *   comb = Sinkhorn of row softmax of fma(mix[8+4i+k]*rstd, scale[2], base[8+4i+k])
 *          (entries fma(e, 1/sum e, sinkhorn_eps)), sigmoid(v) = 1/min(1+exp(-v), 2^126)
 *   li[h] = bf16(fma chain of pre[j]*residual[j][h]), rstd_li = rsqrt(sum li^2 / H + norm_eps)
 *   layer_input[h] = bf16((li[h]*rstd_li) * norm_w[h])   (li itself when norm_w == NULL)
 * workspace: device scratch of at least mhc_workspace_bytes(T, H) bytes.
 */
mhc_status mhc_pre(const uint16_t *residual, const void *weight, const float *scale,
                   const float *base, const void *norm_w, mhc_dtype norm_dtype,
                   const mhc_params *params, int64_t tokens, int hidden,
                   uint16_t *layer_input, float *pre_out, float *post_out,
                   float *comb_out, void *workspace, size_t workspace_bytes,
                   void *stream);

/*
 * Fused post + pre boundary ("mhc_boundary" page, mhc_shifted_post_pre_boundary
 * and MhcBoundaryKernel): the residual update of mhc_post, then the pre of
 * mhc_pre computed on the UPDATED residual.
 * pre_lag: [T, 4] fp32 pre of the previous boundary (shifted form: the layer
 * input collapses the updated residual with pre_lag, all in one pass over
 * the residual), or NULL (unshifted form: it collapses with this boundary's
 * own pre_out, which re-reads the updated residual).
 * Other arguments as in mhc_post and mhc_pre. residual_out may be == residual.
 * Limits of the shifted form: its blocks wait on one another within one
 * launch, so every hidden slice of a 128-token tile must be resident at
 * once, and an item's collapse must fit its tensor-memory buffer. H / 32
 * must therefore have a divisor d <= 8 with H / (32 d) <= 152 (slices of d
 * chunks of 32, at most one per streaming multiprocessor of a GB300): every
 * multiple of 256 up to 38912 qualifies (7168: 28 slices of 256), H = 65536
 * or 32 * 157 does not. Other H return MHC_ERR_UNSUPPORTED before anything
 * is enqueued. The unshifted form has no such limit.
 */
mhc_status mhc_boundary_fused(const uint16_t *x, const uint16_t *residual,
                              const float *post, const float *comb,
                              const float *pre_lag, const void *weight,
                              const float *scale, const float *base,
                              const void *norm_w, mhc_dtype norm_dtype,
                              const mhc_params *params, int64_t tokens, int hidden,
                              uint16_t *residual_out, uint16_t *layer_input,
                              float *pre_out, float *post_out, float *comb_out,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * Unshifted pre from split-K mixes ("The Hyper Connection Preprocessing GPU
 * Kernel Study", the pure path: "square sum and RMSNorm" path 1 and
 * "explaining split-K"): a previous GEMM split the 4H-long contraction of the
 * flattened residual with fn into n_splits parts and left
 *   dot_mix [n_splits, T, 24] fp32   partial mixes (no TF32 rounding implied),
 *   sqrsum  [n_splits, T]     fp32   partial sums of squares of the residual.
 * mix = sum of the splits, ssq = sum of the splits (each in split order, in
 * fp32); rstd = rsqrt(ssq / 4H + hc_norm_eps); pre / post / comb as in
 * mhc_pre; layer_input = the collapse of residual [T, 4, H] with this pre,
 * RMS-normed with norm_w (or the raw collapse when norm_w is NULL).
 * n_splits in [1, 64] (the page's kernel takes 1, 2, 4, 8 or 16), else
 * MHC_ERR_SHAPE. No workspace. Outputs as in mhc_pre; none may alias an
 * input. Enqueued on `stream`: one kernel for up to 1024 tokens (the collapse
 * overlapping the coefficients), else two (coefficients, then the collapse);
 * always two when params->batch_invariant is set.
 */
mhc_status mhc_pre_split_k(const uint16_t *residual, const float *dot_mix, const float *sqrsum,
                           int n_splits, const float *scale, const float *base,
                           const void *norm_w, mhc_dtype norm_dtype, const mhc_params *params,
                           int64_t tokens, int hidden, uint16_t *layer_input, float *pre_out,
                           float *post_out, float *comb_out, void *stream);

/* ---------------------------------------------------------------------- */
/* Allocation-free variant. The pages this library follows have no          */
/* counterpart of this entry point.                                         */

/*
 * mhc_boundary_fused without a workspace, for callers that cannot allocate
 * device memory: code running where cudaMalloc is not permitted or not
 * wanted, such as a serving engine whose memory planner owns every device
 * allocation, or a latency-critical loop that cannot afford the implicit
 * device synchronisation of cudaMalloc/cudaFree. Arguments and results are
 * those of mhc_boundary_fused.
 *
 * Scratch: a fixed 4 MiB array in the library's own device memory, which
 * every GPU that loads the library keeps until the process exits. A call
 * whose mhc_workspace_bytes(tokens, hidden) exceeds 4 MiB returns
 * MHC_ERR_WORKSPACE without enqueuing anything (every decode batch of up to
 * 128 tokens at hidden up to 8192 fits).
 * Set-up: the first call on a device, with that device current, looks up
 * the array's device address; make that first call before any stream
 * capture. Sharing: every call on a device uses the same array and leaves
 * its contents behind; calls that can overlap on the GPU (unordered streams,
 * concurrent host threads) race on it and must be serialised by the caller.
 * No entry needs to start at zero: each call writes every entry it reads.
 * The call allocates nothing (no cudaMalloc, cudaFree or allocating library
 * routine).
 */
mhc_status mhc_boundary_fused_noalloc(const uint16_t *x, const uint16_t *residual,
                                      const float *post, const float *comb,
                                      const float *pre_lag, const void *weight,
                                      const float *scale, const float *base,
                                      const void *norm_w, mhc_dtype norm_dtype,
                                      const mhc_params *params, int64_t tokens, int hidden,
                                      uint16_t *residual_out, uint16_t *layer_input,
                                      float *pre_out, float *post_out, float *comb_out,
                                      void *stream);

/* ---------------------------------------------------------------------- */
/* Status and diagnostics.                                                  */

/* Synchronises `stream`, then reads and clears the current device's status
 * word. Returns MHC_OK, MHC_ERR_DEVICE_TIMEOUT (a kernel's bounded wait ran
 * out since the last read) or MHC_ERR_CUDA. */
mhc_status mhc_get_device_status(void *stream);

/* Extra detail of the last timeout read by mhc_get_device_status: the wait
 * site id (0 if none). */
int mhc_last_timeout_site(void);

/* Human-readable name of a status. Static storage; never NULL. */
const char *mhc_status_string(mhc_status status);

/* Limit of every device-side wait, in nanoseconds (default 1e9 = 1 s).
 * Applies to launches enqueued after the call. ns == 0 restores the default. */
void mhc_set_wait_timeout_ns(uint64_t ns);

/* Test hook for the bounded-wait machinery: launches one CTA that waits on a
 * shared-memory barrier nothing ever arrives at, under the current limit,
 * so that the wait runs out and the kernel returns. Enqueued on `stream`;
 * read the outcome with mhc_get_device_status(). */
mhc_status mhc_debug_unarmed_wait(void *stream);

/* Benchmark hook: the next mhc_pre / mhc_boundary_fused call made by this
 * host thread records `event` (a cudaEvent_t passed as void*) on its stream
 * right after its streaming kernel and before its finishing kernel (the
 * unshifted forms), so that the two kernels can be timed apart with events;
 * a shifted call is the streaming kernel alone, and the event follows it.
 * Consumed by that call; NULL clears a pending event. */
void mhc_debug_record_between(void *event);

/* Test hook for the coefficients' reciprocal (the "mhc_boundary" page's rcp:
 * hardware approximation plus one Newton-Raphson step): compares it with the
 * correctly rounded fp32 reciprocal for the bit patterns first_bits ..
 * first_bits + count - 1 (no wrap past 0xFFFFFFFF, else MHC_ERR_SHAPE).
 * result: device pointer to two u64, 8-byte aligned, set by the caller to
 * {0, ~0} beforehand; result[0] += the number of differing patterns,
 * result[1] = min(its value, the smallest differing pattern). Enqueued on
 * `stream`. The pages have no counterpart. */
mhc_status mhc_debug_rcp_check(uint32_t first_bits, uint64_t count, unsigned long long *result,
                               void *stream);

/* Test hook for the two forms of the coefficients: from reduced values
 * values [tokens][25] fp32 (24 mixes, then the 4H sum of squares), forms
 * pre / post / comb once with one thread per token and once with 16 lanes
 * per token (the form a single-wave shifted call uses), into out_thread and
 * out_lanes [tokens][24] fp32 (pre 4, post 4, comb 16). The two must be
 * bitwise equal. scale [3], base [24] and params as in mhc_pre; device
 * pointers, 16-byte aligned; outputs must not overlap the inputs or each
 * other. Enqueued on `stream`. The pages have no counterpart. */
mhc_status mhc_debug_coef_check(const float *values, const float *scale, const float *base,
                                const mhc_params *params, int hidden, int64_t tokens,
                                float *out_thread, float *out_lanes, void *stream);

/* Slice plan chosen for (T, H): writes the number of hidden slices and the
 * slice width. For tests and the benchmark's byte accounting. */
mhc_status mhc_plan(int64_t tokens, int hidden, int *n_slices, int *slice_width);

/* Whether a shifted mhc_boundary_fused call of (T, H) on the current device
 * runs on one thread-block cluster ("mhc_boundary" page, MhcBoundaryKernel:
 * the hidden slices of one token tile in one cluster, exchanging partial
 * mixes and sums of squares through distributed shared memory): *ctas = the
 * cluster size (the number of hidden slices), or 0 when the call takes the
 * slice-parallel streaming kernel. A call can take a cluster when it has 1 to
 * 64 tokens, params->batch_invariant is 0, its H / 32 chunks split into at
 * most 16 slices of at most 32 chunks and such a cluster can be resident on
 * the device; by default it does so where that is the faster path (a slice
 * of one chunk; of two chunks for up to 32 tokens; of up to four chunks for
 * up to 16 tokens: hidden sizes up to 2048; at hidden 7168 the slice-parallel
 * kernel, which spreads the work over 112 CTAs instead of 16, is faster).
 * Cluster calls need no workspace contents (a workspace is
 * still passed and checked); after the call its bytes 256 .. 256 + 112 T
 * hold each token's 24 mixes and 4H sum of squares as 28 fp32 (the last
 * three zero). Queries the device once per shape. */
mhc_status mhc_plan_cluster(int64_t tokens, int hidden, int *ctas);

/* Benchmark hook: enable = 0 launches the boundary kernels as plain stream
 * kernels; nonzero (the default) as programmatic dependents of the previous
 * kernel on the stream, whose set-up (barriers, tensor memory, descriptor and
 * weight-tile prefetches into L2) overlaps that kernel's end while every
 * read of global memory waits for its completion ("mhc_boundary" page,
 * griddepcontrol around the kernel's prologue). Process-wide. */
void mhc_debug_set_pdl(int enable);

/* Test hook for the dependent launch: a kernel that lets the next kernel on
 * `stream` start at once, waits delay_ns (at most 1,000,000, else
 * MHC_ERR_SHAPE) and then copies n bf16 values from src to dst (device
 * pointers, 16-byte aligned, not overlapping). The pages have no
 * counterpart. */
mhc_status mhc_debug_delayed_copy(const uint16_t *src, uint16_t *dst, int64_t n,
                                  uint32_t delay_ns, void *stream);

/* Test and benchmark hook for the shifted form's decode path, process-wide:
 * 0 (the default) as described at mhc_plan_cluster; 1 every later call takes
 * the slice-parallel streaming kernel; 2 every call that can take a cluster
 * does. Other values act as 0. */
void mhc_debug_set_decode_path(int path);

/* Benchmark hook: the number of kernels this library has launched in the
 * process so far (every entry point that launches, counted when the launch
 * succeeded; thread-safe, process-wide, never reset). The difference across
 * a timed region is the number of the library's kernels in it. */
uint64_t mhc_debug_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* MHC_H */
