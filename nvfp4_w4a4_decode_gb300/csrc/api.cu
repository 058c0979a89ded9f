// api.cu -- the C ABI (include/nvfp4.h): argument checks, then launches on
// the caller's stream.  No allocation, no synchronisation, no global state
// (the split-K kernel's counters live in the caller's workspace).
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/nvfp4.h"
#include "kernels.cuh"

namespace {

bool aligned(const void* p, uintptr_t a)
{
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

int from_cuda(cudaError_t e)
{
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* nvfp4_status_string(int status)
{
    switch (status) {
    case NVFP4_OK: return "NVFP4_OK";
    case NVFP4_ERR_INVALID_ARG: return "NVFP4_ERR_INVALID_ARG";
    case NVFP4_ERR_UNSUPPORTED: return "NVFP4_ERR_UNSUPPORTED";
    case NVFP4_ERR_CUDA: return "NVFP4_ERR_CUDA";
    default: return "NVFP4_ERR_UNKNOWN";
    }
}

const char* nvfp4_version(void)
{
    return "nvfp4-gb300 0.1.0 sm_103a";
}

int nvfp4_global_scale(const float* t, int64_t count, float* g, void* stream)
{
    if (count < 0 || g == nullptr || (count > 0 && t == nullptr))
        return NVFP4_ERR_INVALID_ARG;
    if (count > 0 && !aligned(t, 16))
        return NVFP4_ERR_INVALID_ARG;
    return from_cuda(nvfp4::launch_global_scale(t, count, g, static_cast<cudaStream_t>(stream)));
}

int nvfp4_pack_weight(const float* w, int64_t n, int64_t k, uint8_t* w_q, uint8_t* w_s,
                      float* w_g, void* stream)
{
    if (n < 0 || k < 0 || (k % 16) != 0 || w_g == nullptr)
        return NVFP4_ERR_INVALID_ARG;
    const bool empty = (n == 0 || k == 0);
    if (!empty && (w == nullptr || w_q == nullptr || w_s == nullptr))
        return NVFP4_ERR_INVALID_ARG;
    if (!empty && (!aligned(w, 16) || !aligned(w_q, 8)))
        return NVFP4_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = nvfp4::launch_global_scale(w, empty ? 0 : n * k, w_g, s);
    if (e != cudaSuccess || empty)
        return from_cuda(e);
    return from_cuda(nvfp4::launch_quantize(w, false, n, k, w_g, w_q, w_s, s));
}

int nvfp4_quantize_act_ex(const void* x, int64_t m, int64_t k, const float* x_g, uint8_t* x_q,
                          uint8_t* x_s, uint32_t options, void* stream)
{
    if (m < 0 || k < 0 || (k % 16) != 0 ||
        (options & ~(uint32_t)(NVFP4_FLAG_PDL | NVFP4_FLAG_X_BF16)) != 0)
        return NVFP4_ERR_INVALID_ARG;
    if (m == 0 || k == 0)
        return NVFP4_OK;
    if (x == nullptr || x_g == nullptr || x_q == nullptr || x_s == nullptr)
        return NVFP4_ERR_INVALID_ARG;
    const bool bf16 = (options & NVFP4_FLAG_X_BF16) != 0;
    if (!aligned(x, bf16 ? 8 : 16) || !aligned(x_q, 8) || !aligned(x_g, 4))
        return NVFP4_ERR_INVALID_ARG;
    return from_cuda(nvfp4::launch_quantize(x, bf16, m, k, x_g, x_q, x_s,
                                            static_cast<cudaStream_t>(stream),
                                            (options & NVFP4_FLAG_PDL) != 0));
}

int nvfp4_quantize_act(const float* x, int64_t m, int64_t k, const float* x_g, uint8_t* x_q,
                       uint8_t* x_s, void* stream)
{
    return nvfp4_quantize_act_ex(x, m, k, x_g, x_q, x_s, 0u, stream);
}

int nvfp4_quantize_act_dynamic(const float* x, int64_t m, int64_t k, float* x_g, uint8_t* x_q,
                               uint8_t* x_s, void* stream)
{
    if (m < 0 || k < 0 || (k % 16) != 0 || x_g == nullptr)
        return NVFP4_ERR_INVALID_ARG;
    if (m > 0 && k > 0 && (x == nullptr || x_q == nullptr || x_s == nullptr ||
                           !aligned(x, 16) || !aligned(x_q, 8) || !aligned(x_g, 4)))
        return NVFP4_ERR_INVALID_ARG;
    const int st = nvfp4_global_scale(x, m * k, x_g, stream);
    if (st != NVFP4_OK)
        return st;
    return nvfp4_quantize_act_ex(x, m, k, x_g, x_q, x_s, 0u, stream);
}

namespace {

// Kernel for a GEMM of this shape and operand alignment (negative status on
// a request that cannot be met).  ws_bytes is the workspace on offer.
int select_kernel(int64_t m, int64_t n, int64_t k, uint32_t options, bool ptrs_ok_fast,
                  bool ptrs_ok_tma, int64_t ws_bytes)
{
    const uint32_t req = options & NVFP4_KERNEL_MASK;
    const bool gemv_ok = nvfp4::gemv_supported(m, k) && ptrs_ok_fast;
    const bool mma_ok = nvfp4::mma_supported(m, k) && ptrs_ok_fast;
    const bool tma_ok = nvfp4::tma_supported(m, n, k) && ptrs_ok_tma;
    switch (req) {
    case NVFP4_KERNEL_AUTO:
        // measured on GB300 over the 8B / 32B decode shapes: at M >= 2 the
        // split-K tensor-core kernel (through the workspace its plan wants
        // when the call offers it, else in its cluster form); the CUDA-core
        // stream at M = 1; for shapes no split-K plan takes, the TMA-fed
        // tensor-core kernel when K fits one CTA, else the register-streaming
        // one
        if (m >= 2 && nvfp4::splitk_shape_ok(m, k) && ptrs_ok_fast &&
            nvfp4::splitk_plan_ok(m, n, k, ws_bytes))
            return (int)NVFP4_KERNEL_SPLITK;
        if (gemv_ok)
            return (int)NVFP4_KERNEL_GEMV;
        if (tma_ok && nvfp4::tma_single_cta_k(m, k))
            return (int)NVFP4_KERNEL_TMA;
        return mma_ok ? (int)NVFP4_KERNEL_MMA : (int)NVFP4_KERNEL_GENERIC;
    case NVFP4_KERNEL_GENERIC: return (int)NVFP4_KERNEL_GENERIC;
    case NVFP4_KERNEL_GEMV: return gemv_ok ? (int)NVFP4_KERNEL_GEMV : -(int)NVFP4_ERR_UNSUPPORTED;
    case NVFP4_KERNEL_MMA: return mma_ok ? (int)NVFP4_KERNEL_MMA : -(int)NVFP4_ERR_UNSUPPORTED;
    case NVFP4_KERNEL_TMA: return tma_ok ? (int)NVFP4_KERNEL_TMA : -(int)NVFP4_ERR_UNSUPPORTED;
    case NVFP4_KERNEL_SPLITK:
        return nvfp4::splitk_shape_ok(m, k) && ptrs_ok_fast &&
                       nvfp4::splitk_plan_ok(m, n, k, ws_bytes)
                   ? (int)NVFP4_KERNEL_SPLITK
                   : -(int)NVFP4_ERR_UNSUPPORTED;
    case NVFP4_KERNEL_TC:
        return nvfp4::tc_shape_ok(m, n, k) && ptrs_ok_tma ? (int)NVFP4_KERNEL_TC
                                                          : -(int)NVFP4_ERR_UNSUPPORTED;
    default: return -(int)NVFP4_ERR_UNSUPPORTED;
    }
}

// Shape and option checks shared by the GEMM entry points (NVFP4_OK to go on).
int check_gemm_args(int64_t m, int64_t n, int64_t k, uint32_t options)
{
    if (m < 0 || n < 0 || k < 0 || (k % 16) != 0)
        return NVFP4_ERR_INVALID_ARG;
    if ((options & ~(uint32_t)(NVFP4_KERNEL_MASK | NVFP4_FLAG_PDL | NVFP4_FLAG_Y_BF16 |
                               NVFP4_FLAG_TEST_WAIT_TIMEOUT | NVFP4_FLAG_W_TILED)) != 0)
        return NVFP4_ERR_INVALID_ARG;
    if ((options & NVFP4_FLAG_TEST_WAIT_TIMEOUT) && (options & NVFP4_KERNEL_MASK) != NVFP4_KERNEL_TMA)
        return NVFP4_ERR_INVALID_ARG;
    // the tile-major weight layout is read by the tensor-core kernel only
    if ((options & NVFP4_FLAG_W_TILED) && (options & NVFP4_KERNEL_MASK) != NVFP4_KERNEL_TC)
        return NVFP4_ERR_INVALID_ARG;
    // M above 8 only on the tensor-core kernel, by request
    if (m > ((options & NVFP4_KERNEL_MASK) == NVFP4_KERNEL_TC ? 32 : 8))
        return NVFP4_ERR_UNSUPPORTED;
    return NVFP4_OK;
}

int gemm(const uint8_t* x_q, const uint8_t* x_s, const float* x_g, const uint8_t* w_q,
         const uint8_t* w_s, const float* w_g, void* y, int64_t m, int64_t n, int64_t k,
         uint32_t options, void* workspace, size_t workspace_bytes, void* stream)
{
    const int chk = check_gemm_args(m, n, k, options);
    if (chk != NVFP4_OK)
        return chk;
    if (workspace == nullptr ? workspace_bytes != 0 : !aligned(workspace, 16))
        return NVFP4_ERR_INVALID_ARG;
    if (m == 0 || n == 0)
        return NVFP4_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool y_bf16 = (options & NVFP4_FLAG_Y_BF16) != 0;
    const size_t y_elem = y_bf16 ? 2 : 4;
    if (y == nullptr || !aligned(y, y_elem))
        return NVFP4_ERR_INVALID_ARG;
    if (k == 0)
        return from_cuda(cudaMemsetAsync(y, 0, y_elem * (size_t)(m * n), s));
    if (x_q == nullptr || x_s == nullptr || x_g == nullptr || w_q == nullptr || w_s == nullptr ||
        w_g == nullptr)
        return NVFP4_ERR_INVALID_ARG;
    if (!aligned(x_q, 8) || !aligned(w_q, 8) || !aligned(x_g, 4) || !aligned(w_g, 4))
        return NVFP4_ERR_INVALID_ARG;
    const bool tiled = (options & NVFP4_FLAG_W_TILED) != 0;
    if (tiled && (!aligned(w_q, 16) || !aligned(w_s, 16)))
        return NVFP4_ERR_INVALID_ARG;
    const bool fast_ptrs = aligned(x_q, 32) && aligned(w_q, 32) && aligned(x_s, 4) &&
                           aligned(w_s, 4);
    const bool tma_ptrs = fast_ptrs && aligned(x_s, 32) && aligned(w_s, 32);
    const int64_t ws_bytes = workspace ? (int64_t)workspace_bytes : 0;
    const int kern = select_kernel(m, n, k, options, tiled ? aligned(x_q, 32) : fast_ptrs,
                                   tiled ? aligned(x_q, 32) && aligned(x_s, 32) : tma_ptrs,
                                   ws_bytes);
    if (kern < 0)
        return -kern;
    const bool pdl = (options & NVFP4_FLAG_PDL) != 0;
    const nvfp4::GemmArgs a = {x_q, x_s, x_g, w_q, w_s, w_g, {y, y_bf16 ? 1 : 0}, (int)m, n, k, s};
    switch (kern) {
    case NVFP4_KERNEL_GEMV:
        return from_cuda(nvfp4::launch_gemm_gemv(a, pdl));
    case NVFP4_KERNEL_MMA:
        return from_cuda(nvfp4::launch_gemm_mma(a, pdl));
    case NVFP4_KERNEL_TMA:
        return from_cuda(nvfp4::launch_gemm_tma(a, pdl, (options & NVFP4_FLAG_TEST_WAIT_TIMEOUT) != 0));
    case NVFP4_KERNEL_SPLITK:
        return from_cuda(nvfp4::launch_gemm_splitk(a, pdl, workspace, ws_bytes));
    case NVFP4_KERNEL_TC:
        return from_cuda(nvfp4::launch_gemm_tc(a, pdl, workspace, ws_bytes, tiled));
    default:
        return from_cuda(nvfp4::launch_gemm_generic(a));
    }
}

}  // namespace

int nvfp4_gemm_select_ws(int64_t m, int64_t n, int64_t k, uint32_t options,
                         size_t workspace_bytes)
{
    if (m < 1 || n < 1 || k < 16 || (k % 16) != 0)
        return -NVFP4_ERR_INVALID_ARG;
    if (m > ((options & NVFP4_KERNEL_MASK) == NVFP4_KERNEL_TC ? 32 : 8))
        return -NVFP4_ERR_UNSUPPORTED;
    return select_kernel(m, n, k, options, true, true, (int64_t)workspace_bytes);
}

int nvfp4_gemm_select(int64_t m, int64_t n, int64_t k, uint32_t options)
{
    return nvfp4_gemm_select_ws(m, n, k, options, 0);
}

int64_t nvfp4_gemm_workspace_size(int64_t m, int64_t n, int64_t k, uint32_t options)
{
    if (m < 1 || n < 1 || k < 16 || (k % 16) != 0)
        return -NVFP4_ERR_INVALID_ARG;
    if (m > ((options & NVFP4_KERNEL_MASK) == NVFP4_KERNEL_TC ? 32 : 8))
        return -NVFP4_ERR_UNSUPPORTED;
    const int kern = select_kernel(m, n, k, options, true, true, INT64_MAX);
    if (kern < 0)
        return kern;
    if (kern == (int)NVFP4_KERNEL_TC)
        return nvfp4::tc_workspace_bytes();
    return kern == (int)NVFP4_KERNEL_SPLITK ? nvfp4::splitk_workspace_bytes(m, n, k) : 0;
}

int nvfp4_gemm_smallm_ex(const uint8_t* x_q, const uint8_t* x_s, const float* x_g,
                         const uint8_t* w_q, const uint8_t* w_s, const float* w_g, void* y,
                         int64_t m, int64_t n, int64_t k, uint32_t options, void* stream)
{
    return gemm(x_q, x_s, x_g, w_q, w_s, w_g, y, m, n, k, options, nullptr, 0, stream);
}

int nvfp4_gemm_smallm_ws(const uint8_t* x_q, const uint8_t* x_s, const float* x_g,
                         const uint8_t* w_q, const uint8_t* w_s, const float* w_g, void* y,
                         int64_t m, int64_t n, int64_t k, uint32_t options, void* workspace,
                         size_t workspace_bytes, void* stream)
{
    return gemm(x_q, x_s, x_g, w_q, w_s, w_g, y, m, n, k, options, workspace, workspace_bytes,
                stream);
}

int nvfp4_linear_ws(const void* x, int64_t m, int64_t n, int64_t k, const float* x_g,
                    const uint8_t* w_q, const uint8_t* w_s, const float* w_g, void* y,
                    uint8_t* x_q, uint8_t* x_s, uint32_t options, void* workspace,
                    size_t workspace_bytes, void* stream)
{
    if (m < 0 || n < 0 || k < 0 || (k % 16) != 0)
        return NVFP4_ERR_INVALID_ARG;
    if ((options & ~(uint32_t)(NVFP4_KERNEL_MASK | NVFP4_FLAG_PDL | NVFP4_FLAG_FUSED_QUANTIZE |
                               NVFP4_FLAG_X_BF16 | NVFP4_FLAG_Y_BF16)) != 0)
        return NVFP4_ERR_INVALID_ARG;
    if (m > 8)
        return NVFP4_ERR_UNSUPPORTED;
    if (workspace == nullptr ? workspace_bytes != 0 : !aligned(workspace, 16))
        return NVFP4_ERR_INVALID_ARG;
    if (m == 0 || n == 0)
        return NVFP4_OK;
    const bool x_bf16 = (options & NVFP4_FLAG_X_BF16) != 0;
    const bool y_bf16 = (options & NVFP4_FLAG_Y_BF16) != 0;
    // the fused prologue reads FP32 activations: BF16 input takes two launches
    const bool fuse = (options & NVFP4_FLAG_FUSED_QUANTIZE) != 0 && !x_bf16;
    options &= ~(uint32_t)(NVFP4_FLAG_FUSED_QUANTIZE | NVFP4_FLAG_X_BF16);
    if (k > 0 && (x == nullptr || x_q == nullptr || x_s == nullptr ||
                  !aligned(x, x_bf16 ? 8 : 16) || !aligned(x_q, 8)))
        return NVFP4_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool pdl = (options & NVFP4_FLAG_PDL) != 0;
    if (fuse && k > 0 && w_q != nullptr && w_s != nullptr && w_g != nullptr && x_g != nullptr &&
        y != nullptr && aligned(y, y_bf16 ? 2 : 4) && aligned(x_g, 4) && aligned(w_g, 4)) {
        const bool fast_ptrs = aligned(x_q, 32) && aligned(w_q, 32) && aligned(x_s, 4) &&
                               aligned(w_s, 4);
        const bool tma_ptrs = fast_ptrs && aligned(x_s, 32) && aligned(w_s, 32);
        const int64_t ws_bytes = workspace ? (int64_t)workspace_bytes : 0;
        const int kern = select_kernel(m, n, k, options, fast_ptrs, tma_ptrs, ws_bytes);
        if (kern < 0)
            return -kern;
        if (kern == (int)NVFP4_KERNEL_GEMV) {
            const nvfp4::GemmArgs a = {x_q, x_s, x_g, w_q, w_s, w_g, {y, y_bf16 ? 1 : 0},
                                       (int)m, n, k, s};
            const nvfp4::FusedAct fa = {static_cast<const float*>(x), x_q, x_s};
            return from_cuda(nvfp4::launch_gemm_gemv(a, pdl, &fa));
        }
    }
    const int st = nvfp4_quantize_act_ex(
        x, m, k, x_g, x_q, x_s, (pdl ? NVFP4_FLAG_PDL : 0u) | (x_bf16 ? NVFP4_FLAG_X_BF16 : 0u),
        stream);
    if (st != NVFP4_OK)
        return st;
    return gemm(x_q, x_s, x_g, w_q, w_s, w_g, y, m, n, k, options, workspace, workspace_bytes,
                stream);
}

int nvfp4_linear(const float* x, int64_t m, int64_t n, int64_t k, const float* x_g,
                 const uint8_t* w_q, const uint8_t* w_s, const float* w_g, float* y,
                 uint8_t* x_q, uint8_t* x_s, uint32_t options, void* stream)
{
    return nvfp4_linear_ws(x, m, n, k, x_g, w_q, w_s, w_g, y, x_q, x_s, options, nullptr, 0,
                           stream);
}

int nvfp4_gemm_smallm_static(const uint8_t* x_q, const uint8_t* x_s, const float* x_g,
                             const uint8_t* w_q, const uint8_t* w_s, const float* w_g, void* y,
                             int64_t m, int64_t n, int64_t k, uint32_t options, void* stream)
{
    const uint32_t req = options & NVFP4_KERNEL_MASK;
    if (req != NVFP4_KERNEL_AUTO && req != NVFP4_KERNEL_SPLITK)
        return NVFP4_ERR_INVALID_ARG;
    if ((options & ~(uint32_t)(NVFP4_KERNEL_MASK | NVFP4_FLAG_PDL | NVFP4_FLAG_Y_BF16)) != 0)
        return NVFP4_ERR_INVALID_ARG;
    const bool y_bf16 = (options & NVFP4_FLAG_Y_BF16) != 0;
    const int chk = check_gemm_args(m, n, k, options);
    if (chk != NVFP4_OK)
        return chk;
    if (m == 0 || n == 0)
        return NVFP4_OK;
    if (y == nullptr || x_q == nullptr || x_s == nullptr || x_g == nullptr || w_q == nullptr ||
        w_s == nullptr || w_g == nullptr)
        return NVFP4_ERR_INVALID_ARG;
    if (!aligned(y, y_bf16 ? 2 : 4) || !aligned(x_g, 4) || !aligned(w_g, 4))
        return NVFP4_ERR_INVALID_ARG;
    if (!aligned(x_q, 32) || !aligned(w_q, 32) || !aligned(x_s, 4) || !aligned(w_s, 4))
        return NVFP4_ERR_UNSUPPORTED;
    if (!nvfp4::splitk_shape_ok(m, k) || !nvfp4::splitk_static_fits(m, n, k))
        return NVFP4_ERR_UNSUPPORTED;
    const nvfp4::GemmArgs a = {x_q, x_s, x_g, w_q, w_s, w_g, {y, y_bf16 ? 1 : 0}, (int)m, n, k,
                               static_cast<cudaStream_t>(stream)};
    return from_cuda(nvfp4::launch_gemm_splitk_static(a, (options & NVFP4_FLAG_PDL) != 0));
}

int64_t nvfp4_gemm_static_scratch_bytes(void)
{
    return nvfp4::splitk_static_scratch_bytes();
}

namespace {

// Engine of a multi-linear call: the tensor-core kernel (M up to 32) or the
// CUDA-core stream (M of 1 or 2).  AUTO takes the tensor cores at every M:
// on the 8B-shaped decode step measured on GB300 they stream faster than the
// CUDA-core kernel at M = 1 too (0.668 against 0.697 ms a step).
int chain_engine(int64_t m, uint32_t options)
{
    const uint32_t req = options & NVFP4_KERNEL_MASK;
    (void)m;
    if (req == NVFP4_KERNEL_AUTO)
        return (int)NVFP4_KERNEL_TC;
    if (req == NVFP4_KERNEL_GEMV || req == NVFP4_KERNEL_TC)
        return (int)req;
    return -1;
}

// Checks of a multi-linear call; on success the host descriptions of its
// linears with n >= 1 (linears with n == 0 compute nothing and are dropped).
int check_chain(const nvfp4_chain_linear* linears, int64_t count, int64_t m, uint32_t options,
                bool quantize, int engine, nvfp4::ChainLinear* out, int64_t* kept)
{
    const bool x_bf16 = (options & NVFP4_FLAG_X_BF16) != 0;
    const bool y_bf16 = (options & NVFP4_FLAG_Y_BF16) != 0;
    const bool tc = engine == (int)NVFP4_KERNEL_TC;
    const bool tiled = (options & NVFP4_FLAG_W_TILED) != 0;
    *kept = 0;
    for (int64_t i = 0; i < count; ++i) {
        const nvfp4_chain_linear& L = linears[i];
        if (L.n < 0 || L.k < 0 || (L.k % 16) != 0)
            return NVFP4_ERR_INVALID_ARG;
        if (L.n == 0)
            continue;
        if (!(tc ? nvfp4::tc_shape_ok(m, L.n, L.k) : nvfp4::chain_shape_ok(m, L.n, L.k)))
            return NVFP4_ERR_UNSUPPORTED;
        if (L.x_q == nullptr || L.x_s == nullptr || L.x_g == nullptr || L.w_q == nullptr ||
            L.w_s == nullptr || L.w_g == nullptr || L.y == nullptr ||
            (quantize && L.x == nullptr))
            return NVFP4_ERR_INVALID_ARG;
        const uintptr_t sal = tc ? 16 : 4;  // the tensor-core kernel loads scales 16 bytes at a time
        if (!aligned(L.x_q, 32) || !aligned(L.w_q, tiled ? 16 : 32) || !aligned(L.x_s, sal) ||
            !aligned(L.w_s, sal) || !aligned(L.x_g, 4) || !aligned(L.w_g, 4) ||
            !aligned(L.y, y_bf16 ? 2 : 4) || (quantize && !aligned(L.x, x_bf16 ? 8 : 16)))
            return NVFP4_ERR_INVALID_ARG;
        out[*kept] = {L.x, L.x_g, L.x_q, L.x_s, L.w_q, L.w_s, L.w_g, L.y, L.n, L.k};
        ++*kept;
    }
    return NVFP4_OK;
}

int chain(const nvfp4_chain_linear* linears, int64_t count, int64_t m, uint32_t options,
          void* workspace, size_t workspace_bytes, void* stream, bool quantize)
{
    if (workspace == nullptr ? workspace_bytes != 0 : !aligned(workspace, 16))
        return NVFP4_ERR_INVALID_ARG;
    const uint32_t allowed = NVFP4_KERNEL_MASK | NVFP4_FLAG_PDL | NVFP4_FLAG_Y_BF16 |
                             NVFP4_FLAG_W_TILED | (quantize ? NVFP4_FLAG_X_BF16 : 0u);
    if (count < 0 || m < 0 || (count > 0 && linears == nullptr) || (options & ~allowed) != 0)
        return NVFP4_ERR_INVALID_ARG;
    const int engine = chain_engine(m, options);
    if (engine < 0)
        return NVFP4_ERR_UNSUPPORTED;
    if ((options & NVFP4_FLAG_W_TILED) && engine != (int)NVFP4_KERNEL_TC)
        return NVFP4_ERR_INVALID_ARG;  // the tile-major layout is the tensor-core kernel's
    if (m > (engine == (int)NVFP4_KERNEL_TC ? 32 : 2))
        return NVFP4_ERR_UNSUPPORTED;
    if (count == 0 || m == 0)
        return NVFP4_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool pdl = (options & NVFP4_FLAG_PDL) != 0;
    const int64_t per = engine == (int)NVFP4_KERNEL_TC ? nvfp4::kTcMaxItems : nvfp4::kChainMaxItems;
    // one launch (or launch pair) per `per` linears, all checked first
    nvfp4::ChainLinear part[nvfp4::kChainMaxItems];
    for (int64_t i0 = 0; i0 < count; i0 += per) {
        const int64_t cnt = count - i0 < per ? count - i0 : per;
        int64_t kept = 0;
        const int st = check_chain(linears + i0, cnt, m, options, quantize, engine, part, &kept);
        if (st != NVFP4_OK)
            return st;
    }
    for (int64_t i0 = 0; i0 < count; i0 += per) {
        const int64_t cnt = count - i0 < per ? count - i0 : per;
        int64_t kept = 0;
        check_chain(linears + i0, cnt, m, options, quantize, engine, part, &kept);
        if (kept == 0)
            continue;
        const bool xb = (options & NVFP4_FLAG_X_BF16) != 0, yb = (options & NVFP4_FLAG_Y_BF16) != 0;
        const cudaError_t e =
            engine == (int)NVFP4_KERNEL_TC
                ? nvfp4::launch_tc_chain(part, (int)kept, (int)m, quantize, xb, yb, s, pdl || i0 > 0,
                                         workspace, (int64_t)workspace_bytes,
                                         (options & NVFP4_FLAG_W_TILED) != 0)
                : nvfp4::launch_linear_chain(part, (int)kept, (int)m, quantize, xb, yb, s,
                                             pdl || i0 > 0);
        if (e != cudaSuccess)
            return NVFP4_ERR_CUDA;
    }
    return NVFP4_OK;
}

}  // namespace

int nvfp4_linear_chain(const nvfp4_chain_linear* linears, int64_t count, int64_t m,
                       uint32_t options, void* stream)
{
    return chain(linears, count, m, options, nullptr, 0, stream, true);
}

int nvfp4_gemm_chain(const nvfp4_chain_linear* linears, int64_t count, int64_t m,
                     uint32_t options, void* stream)
{
    return chain(linears, count, m, options, nullptr, 0, stream, false);
}

int nvfp4_linear_chain_ws(const nvfp4_chain_linear* linears, int64_t count, int64_t m,
                          uint32_t options, void* workspace, size_t workspace_bytes, void* stream)
{
    return chain(linears, count, m, options, workspace, workspace_bytes, stream, true);
}

int nvfp4_gemm_chain_ws(const nvfp4_chain_linear* linears, int64_t count, int64_t m,
                        uint32_t options, void* workspace, size_t workspace_bytes, void* stream)
{
    return chain(linears, count, m, options, workspace, workspace_bytes, stream, false);
}

int64_t nvfp4_chain_workspace_size(int64_t m, uint32_t options)
{
    if (m < 1 || (options & ~(uint32_t)(NVFP4_KERNEL_MASK | NVFP4_FLAG_PDL | NVFP4_FLAG_X_BF16 |
                                        NVFP4_FLAG_Y_BF16)) != 0)
        return -NVFP4_ERR_INVALID_ARG;
    const int engine = chain_engine(m, options);
    if (engine < 0 || m > (engine == (int)NVFP4_KERNEL_TC ? 32 : 2))
        return -NVFP4_ERR_UNSUPPORTED;
    return engine == (int)NVFP4_KERNEL_TC ? nvfp4::tc_workspace_bytes() : 0;
}

int64_t nvfp4_tiled_weight_bytes(int64_t n, int64_t k, int64_t* scale_bytes)
{
    if (n < 0 || k < 0 || k % 256 != 0)
        return -NVFP4_ERR_INVALID_ARG;
    if (scale_bytes != nullptr)
        *scale_bytes = nvfp4::tiled_scale_bytes(n, k);
    return nvfp4::tiled_code_bytes(n, k);
}

int nvfp4_tile_weight(const uint8_t* w_q, const uint8_t* w_s, int64_t n, int64_t k, uint8_t* t_q,
                      uint8_t* t_s, void* stream)
{
    if (n < 0 || k < 0 || k % 256 != 0)
        return NVFP4_ERR_INVALID_ARG;
    if (n == 0 || k == 0)
        return NVFP4_OK;
    if (w_q == nullptr || w_s == nullptr || t_q == nullptr || t_s == nullptr ||
        !aligned(w_q, 16) || !aligned(w_s, 16) || !aligned(t_q, 16) || !aligned(t_s, 16))
        return NVFP4_ERR_INVALID_ARG;
    return from_cuda(nvfp4::launch_tile_weight(w_q, w_s, n, k, t_q, t_s,
                                               static_cast<cudaStream_t>(stream)));
}

int nvfp4_chain_supported(int64_t m, int64_t n, int64_t k)
{
    return nvfp4::chain_shape_ok(m, n, k) || nvfp4::tc_shape_ok(m, n, k) ? 1 : 0;
}

int nvfp4_read_probe(const void* buf, int64_t bytes, uint64_t* sink, void* stream)
{
    if (bytes < 0 || bytes % 16 != 0 || sink == nullptr || !aligned(sink, 8) ||
        (bytes > 0 && (buf == nullptr || !aligned(buf, 16))))
        return NVFP4_ERR_INVALID_ARG;
    return from_cuda(nvfp4::launch_read_probe(buf, bytes,
                                              reinterpret_cast<unsigned long long*>(sink),
                                              static_cast<cudaStream_t>(stream)));
}

int nvfp4_device_status(void* stream, uint32_t* flags, int clear)
{
    if (flags == nullptr)
        return NVFP4_ERR_INVALID_ARG;
    unsigned v = 0u;
    const cudaError_t e = nvfp4::read_device_status(static_cast<cudaStream_t>(stream), &v, clear != 0);
    if (e != cudaSuccess)
        return NVFP4_ERR_CUDA;
    *flags = v;
    return NVFP4_OK;
}

int nvfp4_gemm_smallm(const uint8_t* x_q, const uint8_t* x_s, const float* x_g,
                      const uint8_t* w_q, const uint8_t* w_s, const float* w_g, float* y,
                      int64_t m, int64_t n, int64_t k, void* stream)
{
    return nvfp4_gemm_smallm_ex(x_q, x_s, x_g, w_q, w_s, w_g, y, m, n, k, 0u, stream);
}

}  // extern "C"
