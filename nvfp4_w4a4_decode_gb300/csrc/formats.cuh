// formats.cuh -- device-side NVFP4 element codecs for sm_103a.
//
// NVFP4 as used by the W4A4 decode linear ("ReSET: Accurate Latency-Critical
// NVFP4 Reasoning via Step-Aware Temperature Scaling", README "Core
// components" item 2): E2M1 codes (two per byte, low nibble first), one E4M3
// scale per 16 elements along K, one FP32 tensor scale.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace nvfp4 {

// E2M1 round-to-nearest-even of v, saturating at 6, sign kept (also for a
// magnitude that rounds to 0).  Each comparison adds one step of the grid
// 0, .5, 1, 1.5, 2, 3, 4, 6; the midpoints 0.25, 1.25, 2.5 and 5 round down
// (to the even code below) and 0.75, 1.75, 3.5 round up (to the even code
// above), which is where ">" and ">=" alternate.
__device__ __forceinline__ uint32_t e2m1_rne(float v)
{
    const float a = fabsf(v);
    uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f)
               + (a > 2.5f) + (a >= 3.5f) + (a > 5.0f);
    return c | ((__float_as_uint(v) >> 28) & 8u);
}

// E4M3 (FN) round-to-nearest-even of s >= 0, saturating at 448 (code 0x7E),
// through the hardware FP32 -> FP8 conversion with .satfinite.
__device__ __forceinline__ uint32_t e4m3_rne_satfinite(float s)
{
    return (uint32_t)__nv_cvt_float_to_fp8(s, __NV_SATFINITE, __NV_E4M3);
}

// E4M3 byte -> FP32 (exact).
__device__ __forceinline__ float e4m3_to_float(uint32_t code)
{
    __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)code, __NV_E4M3);
    return __half2float(__half(h));
}

// Eight E2M1 codes (one 32-bit word, element 0 in the low nibble) -> four
// f16x2 registers holding elements {0,1}, {2,3}, {4,5}, {6,7}, exact.  The
// word is split into its four bytes by a vector move and each byte goes
// through the hardware E2M1x2 -> f16x2 conversion; the byte split costs no
// extra instructions this way (shifting and masking each byte first more than
// doubled the decode cost when measured).
__device__ __forceinline__ void e2m1x8_to_f16(uint32_t w, uint32_t (&h)[4])
{
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Sum of the two halves of an f16x2, in FP32 (exact: each half converts
// exactly and the sum of two halves fits FP32).
__device__ __forceinline__ float f16x2_sum(uint32_t h)
{
    __half2 v = *reinterpret_cast<__half2*>(&h);
    float2 f = __half22float2(v);
    return f.x + f.y;
}

// Read-only, no-L1-allocate 128-bit load for the weight stream (each weight
// byte is used once).
__device__ __forceinline__ uint4 ld_stream_u4(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ uint2 ld_stream_u2(const void* p)
{
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// ---- the quantisation recipe, shared by every kernel that quantises ----------
// (one implementation, so the stand-alone quantiser and the GEMM prologues
// produce the same bytes)

// Block scale: sc = E4M3 RNE (bmax / (6 g)) saturating, 0 when 6 g == 0;
// returns sc and sets S = dec(sc) * g (FP32, each op correctly rounded).
__device__ __forceinline__ uint32_t block_scale(float bmax, float g, float& S)
{
    const float six_g = __fmul_rn(6.0f, g);
    uint32_t sc = 0;
    if (six_g > 0.0f)
        sc = e4m3_rne_satfinite(__fdiv_rn(bmax, six_g));
    S = __fmul_rn(e4m3_to_float(sc), g);
    return sc;
}

// E2M1 code of t in a block with scale S: RNE of t / S (IEEE division), or the
// signed zero when S == 0.
__device__ __forceinline__ uint32_t element_code(float t, float S)
{
    return (S == 0.0f) ? ((__float_as_uint(t) >> 28) & 8u) : e2m1_rne(__fdiv_rn(t, S));
}

// The 16 elements of a block share S, so the quotients t / S can use one
// reciprocal: r = RN(1/S) (__frcp_rn), q0 = RN(t r), rem = t - S q0 (exact
// with one FMA), q = RN(q0 + rem r).  This is Markstein's FMA correction (P.
// Markstein, "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990): with a correctly rounded
// reciprocal and no intermediate overflow or underflow, q equals the
// correctly rounded quotient, so the codes equal those of element_code().
// The guard keeps S and t inside that domain and falls back to the IEEE
// division outside it; tests compare both forms at every code threshold.
struct BlockDivisor {
    float S, r;
    bool fast;
};

__device__ __forceinline__ BlockDivisor make_divisor(float S)
{
    BlockDivisor d;
    d.S = S;
    d.r = __frcp_rn(S);
    d.fast = S >= 0x1p-100f && S <= 0x1p+100f;
    return d;
}

__device__ __forceinline__ uint32_t element_code_div(float t, const BlockDivisor& d)
{
    if (d.S == 0.0f)
        return (__float_as_uint(t) >> 28) & 8u;
    if (!d.fast || !(fabsf(t) <= 0x1p+100f))
        return e2m1_rne(__fdiv_rn(t, d.S));
    const float q0 = __fmul_rn(t, d.r);
    const float rem = __fmaf_rn(-d.S, q0, t);
    return e2m1_rne(__fmaf_rn(rem, d.r, q0));
}

// Quantise one 16-element block held by one thread: scale code returned,
// codes packed two per byte (element 2j low nibble) into two words.
__device__ __forceinline__ uint32_t quantize_block16(const float* v, float g, uint32_t& w0,
                                                     uint32_t& w1)
{
    float bmax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i)
        bmax = fmaxf(bmax, fabsf(v[i]));
    float S;
    const uint32_t sc = block_scale(bmax, g, S);
    const BlockDivisor d = make_divisor(S);
    w0 = 0u;
    w1 = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        w0 |= element_code_div(v[i], d) << (4 * i);
        w1 |= element_code_div(v[8 + i], d) << (4 * i);
    }
    return sc;
}

}  // namespace nvfp4
