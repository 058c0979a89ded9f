// quantize.cu -- NVFP4 quantisation kernels: tensor amax, tensor scale, and
// the per-16-block E4M3 scale + E2M1 round-to-nearest-even encoder used for
// both the offline weight packing and the on-the-fly activation quantisation
// of the W4A4 decode linear ("ReSET: Accurate Latency-Critical NVFP4
// Reasoning via Step-Aware Temperature Scaling", README "Core components"
// item 2 and "Quantize a model to NVFP4").
//
// Every quantised byte has exactly one correct value; the FP32 steps below
// use explicitly rounded intrinsics (__fmul_rn, __fdiv_rn) so no contraction
// or approximate division can change a code.
#include "formats.cuh"
#include "kernels.cuh"
#include "launch_cache.cuh"

namespace nvfp4 {

// amax(|t|) as FP32 bits, folded into *out with an unsigned atomic max (the
// bit pattern of a non-negative float orders like its value).  *out must
// start at 0.
__global__ void __launch_bounds__(256) amax_kernel(const float* __restrict__ t, int64_t count,
                                                   uint32_t* __restrict__ out)
{
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    float a = 0.0f;
    const int64_t nvec = count / 4;
    const float4* t4 = reinterpret_cast<const float4*>(t);
    for (int64_t i = tid; i < nvec; i += stride) {
        float4 v = __ldg(t4 + i);
        a = fmaxf(a, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    for (int64_t i = nvec * 4 + tid; i < count; i += stride)
        a = fmaxf(a, fabsf(__ldg(t + i)));
    uint32_t bits = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(a));
    if ((threadIdx.x & 31) == 0 && bits != 0)
        atomicMax(out, bits);
}

// *g = amax / 2688 in place (2688 = 6 * 448, the largest E2M1 magnitude times
// the largest E4M3 scale).
__global__ void finalize_scale_kernel(float* g)
{
    const float amax = __uint_as_float(*reinterpret_cast<uint32_t*>(g));
    *g = __fdiv_rn(amax, 2688.0f);
}

// Threads per quantiser CTA.  128 threads at 26 registers take 4096
// registers, which a GEMM CTA pair that leaves that many free (the CUDA-core
// stream's register cap) has room for, so the quantiser of the next linear
// becomes resident while the current GEMM still runs.
#ifndef NVFP4_QUANT_THREADS
#define NVFP4_QUANT_THREADS 128
#endif
// Prefetch X into L2 before waiting on its producer (1) or not (0).
#ifndef NVFP4_QUANT_PREFETCH
#define NVFP4_QUANT_PREFETCH 1
#endif
constexpr int kQuantThreads = NVFP4_QUANT_THREADS;

// Four threads per 16-element block (each holds 4 consecutive elements):
// block amax by a quad shuffle, the E4M3 block scale relative to the tensor
// scale, then each thread's 4 E2M1 codes; the quad gathers its 16 codes into
// two 32-bit words.  Blocks are numbered row-major, so a warp reads 512
// contiguous bytes of t and writes 64 contiguous code bytes.  With
// programmatic dependent launch the kernel lets the next kernel (the GEMM)
// launch at once, asks L2 for its slice of t (a hint: L2 is where global
// memory is coherent, so lines fetched before the producer's writes land are
// updated by them, and the loads below come after the wait), then waits for
// the producer of t.  BF16 input is widened to FP32 exactly (a BF16 value is
// the top half of its FP32 bits).
template <bool PDL, bool BF16>
__global__ void __launch_bounds__(kQuantThreads) quantize_kernel(const void* __restrict__ t,
                                                                 int64_t nblocks,
                                                                 const float* __restrict__ g_ptr,
                                                                 uint8_t* __restrict__ q,
                                                                 uint8_t* __restrict__ s)
{
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t b = tid >> 2;
    const int sub = (int)(tid & 3);
    const bool valid = b < nblocks;
    if constexpr (PDL) {
        asm volatile("griddepcontrol.launch_dependents;");
        // one prefetch per 128-byte line of t: 8 threads (FP32) or 16 (BF16)
        if (NVFP4_QUANT_PREFETCH && valid && (tid & (BF16 ? 15 : 7)) == 0)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const char*>(t) +
                                                           tid * (BF16 ? 8 : 16)));
        asm volatile("griddepcontrol.wait;" ::: "memory");
    }

    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (valid) {
        if constexpr (BF16) {
            const uint2 raw = __ldg(reinterpret_cast<const uint2*>(t) + tid);  // 4 BF16, first low
            v = make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                            __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u));
        } else {
            v = __ldg(reinterpret_cast<const float4*>(t) + tid);
        }
    }
    float bmax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    bmax = fmaxf(bmax, __shfl_xor_sync(0xFFFFFFFFu, bmax, 1));
    bmax = fmaxf(bmax, __shfl_xor_sync(0xFFFFFFFFu, bmax, 2));

    float S;
    const uint32_t sc = block_scale(bmax, __ldg(g_ptr), S);

    const float e[4] = {v.x, v.y, v.z, v.w};
    const BlockDivisor d = make_divisor(S);
    uint32_t codes = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        codes |= element_code_div(e[i], d) << (4 * i);
    // lanes sub = 0,1 own codes 0..7 of the block (one word), sub = 2,3 codes 8..15
    uint32_t mine = codes << (16 * (sub & 1));
    const uint32_t word = mine | __shfl_xor_sync(0xFFFFFFFFu, mine, 1);
    if (valid && (sub & 1) == 0)
        reinterpret_cast<uint32_t*>(q)[2 * b + (sub >> 1)] = word;
    if (valid && sub == 0)
        s[b] = (uint8_t)sc;
}

cudaError_t launch_global_scale(const float* t, int64_t count, float* g, cudaStream_t stream)
{
    cudaError_t err = cudaMemsetAsync(g, 0, sizeof(float), stream);
    if (err != cudaSuccess)
        return err;
    if (count > 0) {
        // enough CTAs for every SM a few times over, then a grid-stride loop
        int64_t blocks = (count / 4 + 255) / 256;
        if (blocks < 1)
            blocks = 1;
        const int64_t cap = (int64_t)32 * device_sm_count(current_device());
        if (blocks > cap)
            blocks = cap;
        amax_kernel<<<(unsigned)blocks, 256, 0, stream>>>(t, count, reinterpret_cast<uint32_t*>(g));
        err = cudaGetLastError();
        if (err != cudaSuccess)
            return err;
    }
    finalize_scale_kernel<<<1, 1, 0, stream>>>(g);
    return cudaGetLastError();
}

template <bool BF16>
cudaError_t launch_quantize_t(const void* t, int64_t nblocks, const float* g, uint8_t* q,
                              uint8_t* s, cudaStream_t stream, bool pdl)
{
    const int64_t grid = (4 * nblocks + kQuantThreads - 1) / kQuantThreads;
    if (!pdl) {
        quantize_kernel<false, BF16><<<(unsigned)grid, kQuantThreads, 0, stream>>>(t, nblocks, g,
                                                                                   q, s);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kQuantThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quantize_kernel<true, BF16>, t, nblocks, g, q, s);
}

cudaError_t launch_quantize(const void* t, bool t_bf16, int64_t rows, int64_t k, const float* g,
                            uint8_t* q, uint8_t* s, cudaStream_t stream, bool pdl)
{
    const int64_t nblocks = rows * (k / 16);
    if (nblocks == 0)
        return cudaSuccess;
    return t_bf16 ? launch_quantize_t<true>(t, nblocks, g, q, s, stream, pdl)
                  : launch_quantize_t<false>(t, nblocks, g, q, s, stream, pdl);
}

}  // namespace nvfp4
