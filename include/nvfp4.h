/*
 * nvfp4.h -- C ABI of the GB300 (sm_103a) small-M NVFP4 W4A4 decode linear.
 *
 * The operation is the linear layer of latency-critical autoregressive decode
 * described in "ReSET: Accurate Latency-Critical NVFP4 Reasoning via
 * Step-Aware Temperature Scaling" (abstract; ReSET README, "Core components"
 * item 2: small-M NVFP4 W4A4 decode kernels for M <= 8):
 *
 *     Y[M,N] = X[M,K] . W[N,K]^T,   1 <= M <= 8,
 *
 * with W stored in NVFP4 and X quantised to NVFP4 on the fly.  The pages do
 * not define the bits of NVFP4; this library uses:
 *   - E2M1 element codes (sign, 2 exponent bits, 1 mantissa bit; magnitudes
 *     0, 0.5, 1, 1.5, 2, 3, 4, 6), packed two per byte, element 2j in the low
 *     nibble of byte j;
 *   - one E4M3 ("FN", max 448) scale byte per 16 consecutive elements of K;
 *   - one FP32 tensor scale g = amax(|T|) / 2688 (2688 = 6 * 448).
 * Quantisation of a 16-block with tensor scale g (FP32, each op correctly
 * rounded): s = bmax / (6 g) (0 when 6 g == 0); sc = E4M3 round-to-nearest-
 * even of s, saturating at 448; S = dec(sc) * g; q_i = E2M1 round-to-nearest-
 * even of t_i / S, saturating at 6, sign kept (also for zeros); S == 0 gives
 * signed zero codes.  Decoded: t_i ~= e2m1(q_i) * dec(sc) * g.
 *
 * Layouts (all row-major, no strides, all buffers owned by the caller):
 *   X    float  [M][K]          W    float  [N][K]
 *   x_q  uint8  [M][K/2]        w_q  uint8  [N][K/2]
 *   x_s  uint8  [M][K/16]       w_s  uint8  [N][K/16]
 *   x_g  float  [1]             w_g  float  [1]
 *   Y    float  [M][N]
 *
 * Conventions shared by every entry point:
 *   - Every pointer is DEVICE memory of the current CUDA device.  Nothing is
 *     allocated, freed or synchronised; work is queued on `stream` (a
 *     cudaStream_t; NULL = the legacy default stream) and the call returns
 *     once it is queued.  The library keeps no state between calls; the only
 *     state that outlives a call is in a caller-owned workspace (the _ws
 *     entry points), whose counters every completed call leaves at zero.
 *   - Argument checks run on the host before anything is launched; a failed
 *     check returns NVFP4_ERR_INVALID_ARG or NVFP4_ERR_UNSUPPORTED and
 *     launches nothing.  A launch failure returns NVFP4_ERR_CUDA.
 *   - K must be a multiple of 16.  X and W must be 16-byte aligned, x_q and
 *     w_q 8-byte aligned.  Sizes of zero are legal: nothing is computed,
 *     except that gemm with K == 0 writes zeros to Y.
 *   - Inputs must be finite; NaN or Inf inputs give unspecified codes.
 */
#ifndef NVFP4_GB300_H
#define NVFP4_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1, /* null pointer, bad size, misalignment */
    NVFP4_ERR_UNSUPPORTED = 2, /* M outside 1..8 */
    NVFP4_ERR_CUDA = 3         /* a CUDA launch or runtime call failed */
} nvfp4_status;

/* Human-readable name of a status code (static string, never NULL). */
const char* nvfp4_status_string(int status);

/* Library version, e.g. "nvfp4-gb300 0.1.0 sm_103a". */
const char* nvfp4_version(void);

/*
 * Tensor scale: *g = amax(|t[0..count)|) / 2688 in FP32, written on the
 * device.  This is the NVFP4 per-tensor FP32 scale; the weight path computes
 * it inside nvfp4_pack_weight, and callers use this entry point to calibrate
 * the static activation scale x_g.  count == 0 writes 0.
 *   t      device float[count], 16-byte aligned
 *   g      device float[1], overwritten
 * Launches a 4-byte memset and two kernels.
 */
int nvfp4_global_scale(const float* t, int64_t count, float* g, void* stream);

/*
 * Weight packing (offline step before decode; the pages' reset-quantize
 * step, README "Quantize a model to NVFP4"): quantise W[N][K] with its own
 * tensor scale.
 *   w      device float[n][k]
 *   w_q    device uint8[n][k/2]   out: E2M1 codes
 *   w_s    device uint8[n][k/16]  out: E4M3 block scales
 *   w_g    device float[1]        out: tensor scale amax/2688
 * Launches a memset and three kernels.
 */
int nvfp4_pack_weight(const float* w, int64_t n, int64_t k,
                      uint8_t* w_q, uint8_t* w_s, float* w_g, void* stream);

/*
 * Activation quantisation, on the fly before each linear (the "A4" half of
 * W4A4): quantise X[M][K] with the static tensor scale *x_g.
 *   x      device float[m][k]
 *   x_g    device float[1]        in: activation tensor scale
 *   x_q    device uint8[m][k/2]   out
 *   x_s    device uint8[m][k/16]  out
 * Any m >= 0 is accepted (the GEMM limits M, not this step).  One kernel.
 */
int nvfp4_quantize_act(const float* x, int64_t m, int64_t k, const float* x_g,
                       uint8_t* x_q, uint8_t* x_s, void* stream);

/*
 * Small-M W4A4 linear: Y[m][n] = gX * gW * sum_b dec(x_s[m][b]) dec(w_s[n][b])
 *                                 * sum_{i in b} e2m1(x_q[m][i]) e2m1(w_q[n][i])
 * accumulated in FP32 (results equal the exact sum up to FP32 rounding).
 * This is the decode-time projection the ReSET README's "Core components"
 * item 2 runs for M <= 8 instead of a tensor-core tile that would be at most
 * 8/128 occupied.
 *   x_q, x_s, x_g   activation codes, scales, tensor scale (as above)
 *   w_q, w_s, w_g   weight codes, scales, tensor scale (as above)
 *   y               device float[m][n], overwritten
 * m must be 0..8 (NVFP4_ERR_UNSUPPORTED otherwise).  One kernel launch:
 * the CUDA-core stream at M = 1, the split-K tensor-core kernel at M >= 2
 * (with no workspace, its cluster form sums the K chunks of a tile through
 * distributed shared memory), and, for shapes it cannot take (K not a
 * multiple of 256, or no plan of at most 8 chunks), a TMA-fed or cluster
 * tensor-core kernel.  The result does not depend on the launch order of
 * CTAs: every reduction has a fixed order.  Independent linears run faster
 * as one nvfp4_linear_chain call.
 */
int nvfp4_gemm_smallm(const uint8_t* x_q, const uint8_t* x_s, const float* x_g,
                      const uint8_t* w_q, const uint8_t* w_s, const float* w_g,
                      float* y, int64_t m, int64_t n, int64_t k, void* stream);

/*
 * Options of the _ex entry points: a kernel choice in the low byte, OR-ed
 * with flags.
 *
 * NVFP4_KERNEL_AUTO     the library's choice for the shape (what the plain
 *                       entry points use).
 * NVFP4_KERNEL_GENERIC  the shape-general CUDA-core kernel (any K % 16 == 0).
 * NVFP4_KERNEL_GEMV     the persistent CUDA-core weight-streaming kernel:
 *                       M <= 2, K a multiple of 1024 and at most 32768.
 * NVFP4_KERNEL_MMA      the tensor-core kernel (mma.sync f16, swap-AB, FP32
 *                       accumulation): M <= 8, K a multiple of 256 that the
 *                       kernel can cut into at most 8 cluster ranks.
 * NVFP4_KERNEL_TMA      the tensor-core kernel fed by bulk asynchronous copies
 *                       (cp.async.bulk + mbarrier ring in shared memory):
 *                       M <= 8, K a multiple of 256 (per cluster rank), N
 *                       below 2^30.
 * NVFP4_KERNEL_SPLITK  the split-K tensor-core kernel (mma.sync f16, swap-AB,
 *                       FP32 accumulation) in which every warp streams its own
 *                       (16 rows x K-chunk) work items with no CTA barrier:
 *                       M <= 8, K a multiple of 256.  K is cut into chunks of
 *                       at most 32768 / M elements; when there is more than
 *                       one, the partial tiles are combined in a workspace
 *                       (the _ws entry points; the last partial of a tile to
 *                       arrive sums them) or, when the call offers less
 *                       workspace than the plan wants, the chunks of a tile
 *                       set run as one thread-block cluster of at most 8 CTAs
 *                       that sums the partials through distributed shared
 *                       memory.  Either way the sum is in chunk order:
 *                       results do not depend on timing.
 * NVFP4_KERNEL_TC      the fifth-generation tensor-core kernel: tcgen05.mma
 *                       kind::mxf4nvf4 (the FP4 codes and UE4M3 block scales
 *                       go to the tensor core as they are; FP32 accumulation
 *                       in tensor memory) with the operands swapped -- 128
 *                       weight rows per MMA tile, the activation rows padded
 *                       to 16 or 32 -- weights streamed by TMA through an
 *                       8-stage shared-memory ring, one persistent CTA per SM.
 *                       M up to 32 (this kernel only; M above 8 has to be
 *                       requested by name), K a multiple of 256; one tile of
 *                       128 rows x K per work unit, so a lone call occupies
 *                       ceil(N / 128) SMs.  Results are exact sums up to FP32
 *                       rounding in the tensor core's own order.  With
 *                       tile-major weights (NVFP4_FLAG_W_TILED) at M <= 8
 *                       the last 20 % (M = 8) to 32 % (M = 1) of every
 *                       linear's tiles (rounded, at least one tile left to the
 *                       tcgen05 MMAs) run on other warps of the same SMs
 *                       through mma.sync instead (f16 operands with the block
 *                       scales folded in exactly, FP32 accumulation), so that
 *                       two weight streams run at once.
 *   The GEMV, MMA and SPLITK kernels need x_q/w_q 32-byte and x_s/w_s 4-byte
 *   aligned, the TMA and TC kernels all four 32-byte aligned; a request a
 *   kernel cannot take returns NVFP4_ERR_UNSUPPORTED.
 * NVFP4_FLAG_TEST_WAIT_TIMEOUT  test hook of the TMA kernel: the first stage
 *                       waits for 16 bytes that never come, so its bounded
 *                       wait runs out (after a few microseconds) and the
 *                       kernel records NVFP4_DEVICE_WAIT_TIMEOUT; Y is left
 *                       unspecified.  For testing the timeout path only.
 * NVFP4_FLAG_X_BF16     (activation quantisation, linear) X is BF16 (raw
 *                       bits, uint16 [m][k], 8-byte aligned) instead of FP32;
 *                       each value is widened to FP32 exactly and quantised by
 *                       the same recipe, so the codes equal those of the FP32
 *                       copy of X.
 * NVFP4_FLAG_Y_BF16     (GEMM, linear) Y is BF16 (uint16 [m][n], 2-byte
 *                       aligned): the FP32 result rounded to nearest even.
 * NVFP4_FLAG_W_TILED    (NVFP4_KERNEL_TC GEMMs and tensor-core chains only) w_q
 *                       and w_s are in the tile-major layout written by
 *                       nvfp4_tile_weight, 16-byte aligned, instead of
 *                       row-major: every pipeline stage of the tensor-core
 *                       kernel is then one contiguous 16 KB bulk copy of
 *                       codes instead of 128 strided pieces, its scales one
 *                       contiguous 2 KB block, and at M <= 8 part of the
 *                       tiles go to a second stream (see NVFP4_KERNEL_TC).
 * NVFP4_FLAG_PDL        programmatic dependent launch: the kernel may start
 *                       while the previous kernel on the stream is still
 *                       running and waits for it before it touches anything
 *                       that kernel could have written -- EXCEPT that the GEMM
 *                       streams w_q/w_s before waiting.  Set it only when the
 *                       work queued just before the call does not write the
 *                       weights (true in decode, where weights are constant).
 *                       (The activation quantiser also asks L2 to prefetch x
 *                       before waiting; a prefetch reads nothing into the
 *                       kernel, and x itself is loaded after the wait.)
 */
#define NVFP4_KERNEL_AUTO 0u
#define NVFP4_KERNEL_GENERIC 1u
#define NVFP4_KERNEL_GEMV 2u
#define NVFP4_KERNEL_MMA 3u
#define NVFP4_KERNEL_TMA 4u
#define NVFP4_KERNEL_SPLITK 5u
#define NVFP4_KERNEL_TC 6u
#define NVFP4_KERNEL_MASK 0xFFu
#define NVFP4_FLAG_PDL 0x100u
#define NVFP4_FLAG_FUSED_QUANTIZE 0x200u
#define NVFP4_FLAG_X_BF16 0x400u
#define NVFP4_FLAG_Y_BF16 0x800u
#define NVFP4_FLAG_W_TILED 0x1000u
#define NVFP4_FLAG_TEST_WAIT_TIMEOUT 0x10000u

/* Bits of the device status word (nvfp4_device_status). */
#define NVFP4_DEVICE_WAIT_TIMEOUT 1u

/*
 * Activation quantisation with a dynamic tensor scale (the other reading of
 * "quantised on the fly": the scale comes from this X, not from calibration):
 * *x_g = amax(|X|) / 2688 is computed and written first (as
 * nvfp4_global_scale), then X is quantised with it (as nvfp4_quantize_act).
 *   x_g   device float[1], OUTPUT here
 * Launches a memset and three kernels.
 */
int nvfp4_quantize_act_dynamic(const float* x, int64_t m, int64_t k, float* x_g,
                               uint8_t* x_q, uint8_t* x_s, void* stream);

/* nvfp4_quantize_act with options: NVFP4_FLAG_PDL, NVFP4_FLAG_X_BF16 (x is
 * then BF16, see above). */
int nvfp4_quantize_act_ex(const void* x, int64_t m, int64_t k, const float* x_g,
                          uint8_t* x_q, uint8_t* x_s, uint32_t options, void* stream);

/* nvfp4_gemm_smallm with a kernel choice and flags (see above).  Same
 * arguments, same result up to FP32 rounding order; y is FP32, or BF16 with
 * NVFP4_FLAG_Y_BF16. */
int nvfp4_gemm_smallm_ex(const uint8_t* x_q, const uint8_t* x_s, const float* x_g,
                         const uint8_t* w_q, const uint8_t* w_s, const float* w_g,
                         void* y, int64_t m, int64_t n, int64_t k,
                         uint32_t options, void* stream);

/*
 * Which kernel a GEMM of shape (m, n, k) with suitably aligned operands runs
 * under `options` (one of NVFP4_KERNEL_*), or minus a status code when the
 * shape is invalid or the requested kernel cannot take it.  Host only; the
 * counterpart of the README's "nvfp4r.status()" inspection.
 */
int nvfp4_gemm_select(int64_t m, int64_t n, int64_t k, uint32_t options);

/* nvfp4_gemm_select for a call that offers `workspace_bytes` of workspace
 * (the _ws entry points). */
int nvfp4_gemm_select_ws(int64_t m, int64_t n, int64_t k, uint32_t options,
                         size_t workspace_bytes);

/*
 * Workspace of the _ws entry points: the bytes that the GEMM of shape
 * (m, n, k) under `options` uses on the current device when offered as much
 * as it wants (0 when it needs none), or minus a status code for an invalid
 * shape or request.  Host only.
 *
 * The workspace is caller-owned device memory, 16-byte aligned, that must be
 * ZERO before its first use: its first part holds per-tile arrival counters
 * (the rest partial sums).  Every call that completes leaves the counters at
 * zero again, so zeroing once at allocation is enough, and one workspace can
 * serve calls of any shapes as long as it is always passed with the same
 * size (the counter region's extent depends on the size only).  Calls that
 * can run at the same time (on other streams) must use separate workspaces:
 * two overlapping calls on one workspace race.  A smaller workspace than this
 * size restricts the kernel's plan to one that fits it or needs none (for
 * the split-K kernel: one chunk, or the cluster form; NVFP4_ERR_UNSUPPORTED
 * when none does).
 */
int64_t nvfp4_gemm_workspace_size(int64_t m, int64_t n, int64_t k, uint32_t options);

/* nvfp4_gemm_smallm_ex with a workspace (NULL with 0 bytes for none). */
int nvfp4_gemm_smallm_ws(const uint8_t* x_q, const uint8_t* x_s, const float* x_g,
                         const uint8_t* w_q, const uint8_t* w_s, const float* w_g,
                         void* y, int64_t m, int64_t n, int64_t k, uint32_t options,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * The split-K GEMM without any allocation (the pages have no counterpart to
 * this entry point; it exists for callers that cannot provide a workspace):
 * as nvfp4_gemm_smallm_ws with NVFP4_KERNEL_SPLITK and a workspace of at
 * least nvfp4_gemm_workspace_size() bytes -- same plan, same result bits --
 * except that the scratch is a library-owned static device array of
 * nvfp4_gemm_static_scratch_bytes() (4 MiB) per device.  Its address is
 * looked up once per device, on the first call (looked up again after a
 * launch fails); the counters it holds start at zero because the array is
 * zero when the library loads and every completed call leaves them zero.
 * Nothing is allocated, freed or cleared.
 *   options   NVFP4_KERNEL_AUTO or NVFP4_KERNEL_SPLITK, optionally
 *             NVFP4_FLAG_PDL and NVFP4_FLAG_Y_BF16 (anything else:
 *             NVFP4_ERR_INVALID_ARG)
 * Returns NVFP4_ERR_UNSUPPORTED, launching nothing, when the shape is not
 * one the split-K kernel takes, the operands are not aligned for it, or the
 * scratch the call needs exceeds the static array.  All calls on a device
 * share the one array: calls that may overlap in time (other streams, other
 * host threads without ordering) race and give wrong results; calls on one
 * stream are ordered and safe.
 */
int nvfp4_gemm_smallm_static(const uint8_t* x_q, const uint8_t* x_s, const float* x_g,
                             const uint8_t* w_q, const uint8_t* w_s, const float* w_g,
                             void* y, int64_t m, int64_t n, int64_t k, uint32_t options,
                             void* stream);

/* Bytes of the static scratch array behind nvfp4_gemm_smallm_static. */
int64_t nvfp4_gemm_static_scratch_bytes(void);

/*
 * One W4A4 decode linear: quantise X[m][k] with the static tensor scale *x_g
 * (exactly as nvfp4_quantize_act: the codes and scales are written to x_q and
 * x_s) and compute Y[m][n] = X . W^T from them (as nvfp4_gemm_smallm_ex with
 * `options`): two launches.  With NVFP4_FLAG_FUSED_QUANTIZE, and when the
 * chosen kernel is the CUDA-core stream (M <= 2, K a multiple of 1024), it is
 * ONE kernel instead: each CTA quantises X cooperatively in its prologue (same
 * bytes as the stand-alone quantiser; CTA 0 stores them).  One launch is
 * cheaper for a lone call; inside a CUDA graph with NVFP4_FLAG_PDL the two
 * launches measured faster (the separate quantiser overlaps the previous GEMM,
 * the fused prologue does not), hence the default.  With NVFP4_FLAG_PDL the
 * kernel(s) start streaming weights before the previous kernel on the stream
 * has finished (the weights must not be written by it).
 *   x        device float[m][k], 16-byte aligned
 *   x_q, x_s device outputs as in nvfp4_quantize_act (required)
 *   others   as in nvfp4_gemm_smallm
 */
int nvfp4_linear(const float* x, int64_t m, int64_t n, int64_t k, const float* x_g,
                 const uint8_t* w_q, const uint8_t* w_s, const float* w_g, float* y,
                 uint8_t* x_q, uint8_t* x_s, uint32_t options, void* stream);

/* nvfp4_linear with a workspace for the GEMM (as nvfp4_gemm_smallm_ws) and
 * the dtype flags: NVFP4_FLAG_X_BF16 (x is BF16; the fused one-kernel form is
 * then not used) and NVFP4_FLAG_Y_BF16 (y is BF16). */
int nvfp4_linear_ws(const void* x, int64_t m, int64_t n, int64_t k, const float* x_g,
                    const uint8_t* w_q, const uint8_t* w_s, const float* w_g, void* y,
                    uint8_t* x_q, uint8_t* x_s, uint32_t options, void* workspace,
                    size_t workspace_bytes, void* stream);

/*
 * Many decode linears in one persistent launch.  The decode step of the
 * ReSET README ("Core components" item 2; its trace figure decodes at batch 1
 * under CUDA graphs) is a long sequence of small-M linears.  Launched one by
 * one, each pays a launch, a ramp-up of its weight stream and a tail in which
 * its last CTAs finish alone: a few microseconds per linear, comparable to
 * the DRAM time of an 8B-shaped layer.  These entry points take a list of
 * INDEPENDENT linears -- no linear reads another's output, all activations
 * are ready when the call's work starts (the projections that share one
 * input, the linears of several layers whose inputs are known, experts of a
 * mixture) -- and stream all their weights in one persistent launch (the
 * CUDA-core stream or the tensor-core kernel), whose weight loads do not
 * pause between linears.  On the CUDA-core stream each output equals, bit for
 * bit, that of the single-linear NVFP4_KERNEL_GEMV for the same linear (the
 * same per-output reduction order).  Linears that depend on each other need
 * one call per linear (nvfp4_linear with NVFP4_FLAG_PDL).
 *
 *   x      activations [m][k]: FP32, or BF16 with NVFP4_FLAG_X_BF16
 *          (nvfp4_linear_chain quantises them; nvfp4_gemm_chain ignores x)
 *   x_g    activation tensor scale [1]
 *   x_q    codes [m][k/2] and x_s block scales [m][k/16]: OUTPUTS of
 *          nvfp4_linear_chain, INPUTS of nvfp4_gemm_chain
 *   w_q, w_s, w_g   packed weights as for nvfp4_gemm_smallm
 *   y      output [m][n]: FP32, or BF16 with NVFP4_FLAG_Y_BF16
 *   n, k   n >= 0 (a linear with n == 0 is skipped); k a multiple of 1024,
 *          at most 32768
 * Every pointer is device memory; x_q and w_q 32-byte aligned, x_s and w_s
 * 4-byte, x 16-byte (8 for BF16), y 4-byte (2 for BF16).  The y, x_q and x_s
 * buffers of different linears must not overlap each other or any input of
 * the call (all linears are in flight at once).
 */
typedef struct {
    const void* x;
    const float* x_g;
    uint8_t* x_q;
    uint8_t* x_s;
    const uint8_t* w_q;
    const uint8_t* w_s;
    const float* w_g;
    void* y;
    int64_t n;
    int64_t k;
} nvfp4_chain_linear;

/* Linears per launch: longer lists are cut into launches of this many
 * (CUDA-core stream; tensor-core kernel). */
#define NVFP4_CHAIN_MAX_LINEARS 256
#define NVFP4_TC_MAX_LINEARS 150

/*
 * Quantise every linear's activations (one launch: the recipe of
 * nvfp4_quantize_act, same bytes) and compute every Y (one persistent
 * launch, which starts streaming weights before the codes are written and
 * reads them once they are).  `linears` is a HOST array of `count`
 * descriptions, read during the call only.  options: a kernel choice in the
 * low byte --
 *   NVFP4_KERNEL_AUTO   the tensor-core kernel (measured faster than the
 *                       CUDA-core stream on the decode step at every m);
 *   NVFP4_KERNEL_GEMV   the CUDA-core stream: m of 1 or 2, k a multiple of
 *                       1024 up to 32768 (each output bit-exact with the
 *                       single-linear NVFP4_KERNEL_GEMV);
 *   NVFP4_KERNEL_TC     the tensor-core kernel (NVFP4_KERNEL_TC above): m up
 *                       to 32, k a multiple of 256, x_s and w_s 16-byte
 *                       aligned; NVFP4_TC_MAX_LINEARS linears per launch
 * -- OR-ed with NVFP4_FLAG_PDL (the first launch may start before the
 * previous kernel on the stream ends; the weights must not be written by
 * it), NVFP4_FLAG_X_BF16, NVFP4_FLAG_Y_BF16, NVFP4_FLAG_W_TILED (tensor
 * cores only: every linear's w_q / w_s in the tile-major layout of
 * nvfp4_tile_weight, 16-byte aligned).  Every description is checked
 * before anything is launched: NVFP4_ERR_INVALID_ARG for a null or
 * misaligned pointer or a bad size, NVFP4_ERR_UNSUPPORTED for an m or shape
 * the chosen kernel does not take.  Asynchronous on `stream`; nothing
 * allocated.  The tensor-core kernel's waits are bounded: one that runs out
 * (nothing in a correct call makes that happen) sets
 * NVFP4_DEVICE_WAIT_TIMEOUT (nvfp4_device_status) and leaves Y unspecified.
 */
int nvfp4_linear_chain(const nvfp4_chain_linear* linears, int64_t count, int64_t m,
                       uint32_t options, void* stream);

/* The GEMM half of nvfp4_linear_chain: x_q / x_s are inputs (quantised
 * beforehand), x is not read; one launch per NVFP4_CHAIN_MAX_LINEARS (or
 * NVFP4_TC_MAX_LINEARS) linears.  options: a kernel choice as above,
 * NVFP4_FLAG_PDL, NVFP4_FLAG_Y_BF16. */
int nvfp4_gemm_chain(const nvfp4_chain_linear* linears, int64_t count, int64_t m,
                     uint32_t options, void* stream);

/*
 * The chain entry points with a workspace: the tensor-core kernel then
 * gives every CTA an equal share of the weight stream, cutting 128-row tiles
 * between CTAs where the shares end, and the CTAs that share a tile add
 * their partial sums through the workspace in a fixed order (the last to
 * finish sums them; results do not depend on timing).  Without a workspace
 * the shares end on tile boundaries, which leaves SMs idle when a call has
 * few or large tiles (a lone linear of a few thousand rows, K = 25600).
 *   workspace        caller-owned device memory, 16-byte aligned, ZERO before
 *                    its first use; every completed call leaves it so, and it
 *                    may serve any number of calls that do not overlap in time
 *                    (overlapping calls need separate workspaces)
 *   workspace_bytes  at least nvfp4_chain_workspace_size() (less: no
 *                    workspace is used); NULL with 0 for none
 * The CUDA-core stream takes no workspace (it is ignored).
 */
int nvfp4_linear_chain_ws(const nvfp4_chain_linear* linears, int64_t count, int64_t m,
                          uint32_t options, void* workspace, size_t workspace_bytes, void* stream);
int nvfp4_gemm_chain_ws(const nvfp4_chain_linear* linears, int64_t count, int64_t m,
                        uint32_t options, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Tile-major weight layout of the tensor-core kernel (an offline repack of
 * the row-major packed weights; the bytes are the same, only their order and
 * the zero rows that pad N to a multiple of 128 differ).  For tile t (weight
 * rows 128 t .. 128 t + 127) and stage s (K elements 256 s .. 256 s + 255):
 *   t_q  block (t, s) of 16384 bytes at offset (t * K/256 + s) * 16384: row r
 *        at 128 r, its 16-byte chunk c (K elements 256 s + 32 c ..) at
 *        16 (c XOR (r mod 8)) -- the 128-byte-swizzled image the tensor core
 *        reads from shared memory;
 *   t_s  block (t, s) of 2048 bytes at offset (t * K/256 + s) * 2048: row r's
 *        16 block scales of the stage at 16 r.
 * Rows past n are zero.  nvfp4_tiled_weight_bytes returns the code bytes
 * (ceil(n/128) * 128 * k/2) and writes the scale bytes (ceil(n/128) * 128 *
 * k/16) to *scale_bytes (may be NULL), or minus a status code; k must be a
 * multiple of 256.  nvfp4_tile_weight writes both from w_q [n][k/2] and
 * w_s [n][k/16] (all four pointers 16-byte aligned, device memory; two
 * kernels on `stream`).  Pass the results with NVFP4_FLAG_W_TILED.
 */
int64_t nvfp4_tiled_weight_bytes(int64_t n, int64_t k, int64_t* scale_bytes);
int nvfp4_tile_weight(const uint8_t* w_q, const uint8_t* w_s, int64_t n, int64_t k, uint8_t* t_q,
                      uint8_t* t_s, void* stream);

/* Workspace bytes the chain entry points use with this m and options on the
 * current device (0 for the CUDA-core stream), or minus a status code.  The
 * tensor-core kernel also uses this size through the _ws GEMM entry points
 * (nvfp4_gemm_workspace_size reports it for NVFP4_KERNEL_TC).  Host only. */
int64_t nvfp4_chain_workspace_size(int64_t m, uint32_t options);

/* 1 when a linear of shape (m, n, k) can be part of a chain (on either
 * kernel), else 0.  Host only. */
int nvfp4_chain_supported(int64_t m, int64_t n, int64_t k);

/*
 * Read-only streaming probe, a measurement aid with no counterpart in the
 * method: the DRAM read rate a plain stream of 128-bit loads reaches on this
 * device, the ceiling the GEMM's weight stream is compared with.
 *   buf    device, `bytes` bytes (16-byte aligned; read-only, not owned)
 *   bytes  a multiple of 16 (0: only the sink is written)
 *   sink   device uint64_t[1] (8-byte aligned), OUTPUT: zeroed on the stream,
 *          then the XOR of every 8-byte word of buf (so no load is dropped)
 * Launches a memset and one kernel (every word loaded once, non-allocating
 * in L1); asynchronous on `stream`.  NVFP4_ERR_INVALID_ARG for a negative or
 * ragged size, a null or misaligned pointer.
 */
int nvfp4_read_probe(const void* buf, int64_t bytes, uint64_t* sink, void* stream);

/*
 * Device status word of the library on the current device: the OR of the
 * NVFP4_DEVICE_* bits recorded by kernels since it was last cleared (a wait
 * that ran out of its budget sets NVFP4_DEVICE_WAIT_TIMEOUT; the results of
 * that launch are unspecified).  Synchronises `stream`; with clear != 0 the
 * word is reset to 0 afterwards.  *flags is written on the host.
 */
int nvfp4_device_status(void* stream, uint32_t* flags, int clear);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_GB300_H */
