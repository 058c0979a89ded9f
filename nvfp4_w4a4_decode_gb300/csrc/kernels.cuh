// kernels.cuh -- host-side launchers shared between the translation units of
// the library (the C ABI in api.cu calls these).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nvfp4 {

// Output of a GEMM: FP32, or BF16 rounded to nearest even from the same FP32
// value.
struct OutY {
    void* p;
    int bf16;
};

__device__ __forceinline__ void store_y(const OutY& y, int64_t i, float v)
{
    if (y.bf16)
        reinterpret_cast<__nv_bfloat16*>(y.p)[i] = __float2bfloat16_rn(v);
    else
        reinterpret_cast<float*>(y.p)[i] = v;
}

struct GemmArgs {
    const uint8_t* xq;
    const uint8_t* xs;
    const float* xg;
    const uint8_t* wq;
    const uint8_t* ws;
    const float* wg;
    OutY y;
    int m;
    int64_t n;
    int64_t k;
    cudaStream_t stream;
};

cudaError_t launch_global_scale(const float* t, int64_t count, float* g, cudaStream_t stream);

// t is FP32, or BF16 when t_bf16 (converted exactly before quantising).
cudaError_t launch_quantize(const void* t, bool t_bf16, int64_t rows, int64_t k, const float* g,
                            uint8_t* q, uint8_t* s, cudaStream_t stream, bool pdl = false);

// Any shape with k % 16 == 0 and 8-byte aligned code rows.
cudaError_t launch_gemm_generic(const GemmArgs& a);

// FP32 activations for a GEMM that quantises them in its prologue, and where
// the quantised codes and scales go (both may be null).
struct FusedAct {
    const float* x;
    uint8_t* xq_out;
    uint8_t* xs_out;
};

// Persistent CUDA-core weight-streaming kernel: m in {1, 2}, k a multiple of
// 1024 up to 32768; x_q/w_q 16-byte and x_s/w_s 4-byte aligned.  With `fa`
// the activations are quantised in the prologue (x 16-byte aligned).
bool gemv_supported(int64_t m, int64_t k);
cudaError_t launch_gemm_gemv(const GemmArgs& a, bool pdl, const FusedAct* fa = nullptr);

// Tensor-core (mma.sync f16, swap-AB) kernel: m in 1..8, k a multiple of 256
// that splits into at most 8 cluster ranks of 4..16 warps x 1, 2 or 4
// 256-element ranges; x_q/w_q 32-byte and x_s/w_s 4-byte aligned.
bool mma_supported(int64_t m, int64_t k);
cudaError_t launch_gemm_mma(const GemmArgs& a, bool pdl);

// Tensor-core kernel fed by cp.async.bulk into a shared-memory ring: m in
// 1..8, k a multiple of 256 per cluster rank, n < 2^30; all operand pointers
// 32-byte aligned.  test_timeout arms the bounded-wait test hook.
bool tma_supported(int64_t m, int64_t n, int64_t k);
// true when the TMA kernel keeps the whole K in one CTA (no cluster split)
bool tma_single_cta_k(int64_t m, int64_t k);
cudaError_t launch_gemm_tma(const GemmArgs& a, bool pdl, bool test_timeout);
// Split-K tensor-core kernel, one work stream per warp: m in 1..8, k a
// multiple of 256; x_q/w_q 16-byte and x_s/w_s 2-byte aligned.  When K is cut
// into more than one chunk the partial tiles go through a workspace of
// splitk_workspace_bytes() bytes (the plan with an unlimited workspace); it
// must be zero before its first use and every completed launch leaves it
// zero.  With a smaller workspace (or none) the plan is restricted to what
// fits or needs none (one chunk, or the cluster form: at most 8 chunks as one
// thread-block cluster, partials summed through distributed shared memory);
// splitk_plan_ok() says whether one exists.
bool splitk_shape_ok(int64_t m, int64_t k);
bool splitk_plan_ok(int64_t m, int64_t n, int64_t k, int64_t workspace_bytes);
int64_t splitk_workspace_bytes(int64_t m, int64_t n, int64_t k);
cudaError_t launch_gemm_splitk(const GemmArgs& a, bool pdl, void* workspace,
                               int64_t workspace_bytes);

// The split-K kernel on a library-owned static scratch array of
// splitk_static_scratch_bytes() (no allocation): splitk_static_fits() says
// whether the plan a workspace of any size would get fits in it (then the
// results equal those of launch_gemm_splitk with such a workspace).
int64_t splitk_static_scratch_bytes();
bool splitk_static_fits(int64_t m, int64_t n, int64_t k);
cudaError_t launch_gemm_splitk_static(const GemmArgs& a, bool pdl);

// One linear of a multi-linear launch (host-side description; every pointer
// is device memory).  x is FP32 or BF16 (launch-wide flag); xq / xs are the
// quantised activations (written by the launch's quantiser, or inputs when it
// has none); y is FP32 or BF16 (launch-wide flag).
struct ChainLinear {
    const void* x;
    const float* xg;
    uint8_t* xq;
    uint8_t* xs;
    const uint8_t* wq;
    const uint8_t* ws;
    const float* wg;
    void* y;
    int64_t n;
    int64_t k;
};

// Linears per launch of the multi-linear kernels (their descriptions travel
// in the kernel parameters).
constexpr int kChainMaxItems = 256;

// Whether a linear of this shape can be part of a multi-linear launch: M of
// 1 or 2, K a multiple of 1024 up to 32768, N below 2^30.
bool chain_shape_ok(int64_t m, int64_t n, int64_t k);

// 1 <= count <= kChainMaxItems linears (each with n >= 1) in one persistent
// CUDA-core weight-streaming launch, preceded (quantize) by one launch that
// quantises every linear's activations.  Operands aligned as for the
// single-linear CUDA-core kernel; the y, xq and xs buffers of different
// linears must not overlap.
cudaError_t launch_linear_chain(const ChainLinear* items, int count, int m, bool quantize,
                                bool x_bf16, bool y_bf16, cudaStream_t stream, bool pdl);

// The activation quantisation of up to kChainMaxItems linears in one launch
// (four threads per 16-element block, the stand-alone quantiser's recipe).
// With pdl it may start before the previous kernel on the stream ends (it
// waits before reading x).
cudaError_t launch_chain_quant(const ChainLinear* items, int count, int m, bool x_bf16,
                               cudaStream_t stream, bool pdl);

// Tensor-core (tcgen05, kind::mxf4nvf4) persistent kernel over up to
// kTcMaxItems independent linears: m in 1..32, k a multiple of 256, n below
// 2^30; w_q 16-byte, x_q / x_s / w_s 16-byte aligned.  With quantize, one
// launch of launch_chain_quant comes first.
#ifndef NVFP4_TC_MAX_ITEMS
#define NVFP4_TC_MAX_ITEMS 150
#endif
constexpr int kTcMaxItems = NVFP4_TC_MAX_ITEMS;
constexpr int kTcMaxCtas = 256;
// With a workspace of at least tc_workspace_bytes() (zero before its first
// use; every completed launch leaves its counters zero) the CTAs get equal
// shares of the stages and tiles cut between two CTAs are combined through
// it in a fixed order; without one the shares end on tile boundaries.
bool tc_shape_ok(int64_t m, int64_t n, int64_t k);
int64_t tc_workspace_bytes();
// With tiled, every linear's wq / ws are in the tile-major layout of
// launch_tile_weight (16-byte aligned).
cudaError_t launch_tc_chain(const ChainLinear* items, int count, int m, bool quantize, bool x_bf16,
                            bool y_bf16, cudaStream_t stream, bool pdl, void* workspace = nullptr,
                            int64_t workspace_bytes = 0, bool tiled = false);
// One linear through the tensor-core kernel (m up to 32).
cudaError_t launch_gemm_tc(const GemmArgs& a, bool pdl, void* workspace, int64_t workspace_bytes,
                           bool tiled);

// Tile-major weight layout of the tensor-core kernel: rows padded to a
// multiple of 128; codes as 16 KB blocks (tile, stage of 256 K) holding the
// 128-byte-swizzled shared-memory image, scales as 2 KB blocks (tile, stage)
// of 16 bytes per row.  Sizes in bytes, and the repack from the row-major
// layout (two kernels).
int64_t tiled_code_bytes(int64_t n, int64_t k);
int64_t tiled_scale_bytes(int64_t n, int64_t k);
cudaError_t launch_tile_weight(const uint8_t* wq, const uint8_t* ws, int64_t n, int64_t k,
                               uint8_t* tq, uint8_t* ts, cudaStream_t stream);

cudaError_t read_device_status(cudaStream_t stream, unsigned* out, bool clear);
// Device address of the status word on the current device (for kernels of
// other translation units that record bounded-wait timeouts in it).
cudaError_t device_status_address(unsigned** out);

// Read-only streaming probe: zeroes *sink on the stream, then loads every
// 16-byte word of buf once and XORs all its 8-byte words into *sink.  buf
// 16-byte aligned, bytes a multiple of 16.
cudaError_t launch_read_probe(const void* buf, int64_t bytes, unsigned long long* sink,
                              cudaStream_t stream);

}  // namespace nvfp4
