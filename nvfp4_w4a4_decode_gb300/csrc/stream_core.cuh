// stream_core.cuh -- register-level pieces of the CUDA-core weight stream
// (the broadcast-weight GEMV of the ReSET README, "Core components" item 2),
// shared by the single-linear kernel (gemm_gemv.cu) and the multi-linear
// persistent kernel (gemm_chain.cu).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "formats.cuh"

namespace nvfp4 {

// Read-only, no-L1-allocate 16-bit load (the two E4M3 scales of a thread's
// 32-element chunk).
__device__ __forceinline__ uint32_t ld_u16_nc(const uint8_t* p)
{
    unsigned short v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// Two E4M3 bytes (low 16 bits) -> two floats, exact.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two)
{
    uint32_t h;
    asm("{\n\t.reg .b16 lo;\n\tcvt.u16.u32 lo, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
        : "=r"(h)
        : "r"(two));
    return __half22float2(*reinterpret_cast<__half2*>(&h));
}

// One step of a butterfly reduce-scatter over lanes: lanes with `upper`
// clear keep a (adding the partner's a), lanes with it set keep b.
__device__ __forceinline__ float rs_step(float a, float b, int bit, bool upper)
{
    const float send = upper ? a : b;
    const float keep = upper ? b : a;
    return keep + __shfl_xor_sync(0xFFFFFFFFu, send, bit);
}

// A thread's 32-element chunk of each of the M activation rows, decoded once:
// E2M1 values as f16x2 (unscaled) and the two block scales as floats.
template <int M>
struct XChunk {
    uint32_t h[M][16];
    float s[M][2];
};

template <int M>
__device__ __forceinline__ void load_x_chunk(XChunk<M>& x, const uint8_t* xq, const uint8_t* xs,
                                             int64_t kh, int64_t kb, int c)
{
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(xq + m * kh + 16 * c));
        const uint32_t sc2 = __ldg(reinterpret_cast<const unsigned short*>(xs + m * kb + 2 * c));
        e2m1x8_to_f16(v.x, *reinterpret_cast<uint32_t(*)[4]>(&x.h[m][0]));
        e2m1x8_to_f16(v.y, *reinterpret_cast<uint32_t(*)[4]>(&x.h[m][4]));
        e2m1x8_to_f16(v.z, *reinterpret_cast<uint32_t(*)[4]>(&x.h[m][8]));
        e2m1x8_to_f16(v.w, *reinterpret_cast<uint32_t(*)[4]>(&x.h[m][12]));
        const float2 f = e4m3x2_to_float2(sc2);
        x.s[m][0] = f.x;
        x.s[m][1] = f.y;
    }
}

// The MAC of one 32-element weight chunk (codes `wh` decoded to f16x2,
// scales `sw`) against the M activation chunks: per 16-block and row, 8 packed
// HFMA2 of exact E2M1 products (each f16 half sums 8 products, |sum| <= 288 in
// steps of 1/4, so the block sum is exact), then one FP32 FMA with the
// block's scale product.
template <int M>
__device__ __forceinline__ void mac_chunk(const uint32_t (&wh)[16], float2 sw, const XChunk<M>& x,
                                          float (&acc)[M])
{
#pragma unroll
    for (int m = 0; m < M; ++m) {
        uint32_t p0 = 0u, p1 = 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            p0 = hfma2_u32(wh[j], x.h[m][j], p0);
            p1 = hfma2_u32(wh[8 + j], x.h[m][8 + j], p1);
        }
        acc[m] = fmaf(f16x2_sum(p1), __fmul_rn(x.s[m][1], sw.y),
                      f16x2_sum(p0) * __fmul_rn(x.s[m][0], sw.x));
    }
}

__device__ __forceinline__ void decode_w_chunk(const uint4& w, uint32_t (&wh)[16])
{
    e2m1x8_to_f16(w.x, *reinterpret_cast<uint32_t(*)[4]>(&wh[0]));
    e2m1x8_to_f16(w.y, *reinterpret_cast<uint32_t(*)[4]>(&wh[4]));
    e2m1x8_to_f16(w.z, *reinterpret_cast<uint32_t(*)[4]>(&wh[8]));
    e2m1x8_to_f16(w.w, *reinterpret_cast<uint32_t(*)[4]>(&wh[12]));
}

// Butterfly reduce-scatter of STAGES per-lane values (4, 8 or 16) over a
// warp, then the remaining lane bits summed: afterwards lane l holds the warp
// sum of stage `sidx`, and `writer` is set on one lane per stage.
template <int STAGES>
__device__ __forceinline__ float reduce_scatter(const float (&a)[STAGES], int lane, int& sidx,
                                                bool& writer)
{
    const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4, u2 = lane & 2;
    float v;
    if constexpr (STAGES == 16) {
        float b[8], c[4], d[2];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            b[i] = rs_step(a[i], a[8 + i], 16, u16);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            c[i] = rs_step(b[i], b[4 + i], 8, u8);
#pragma unroll
        for (int i = 0; i < 2; ++i)
            d[i] = rs_step(c[i], c[2 + i], 4, u4);
        v = rs_step(d[0], d[1], 2, u2);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
        sidx = (u16 ? 8 : 0) + (u8 ? 4 : 0) + (u4 ? 2 : 0) + (u2 ? 1 : 0);
        writer = (lane & 1) == 0;
    } else if constexpr (STAGES == 8) {
        const float a0 = rs_step(a[0], a[4], 16, u16);
        const float a1 = rs_step(a[1], a[5], 16, u16);
        const float a2 = rs_step(a[2], a[6], 16, u16);
        const float a3 = rs_step(a[3], a[7], 16, u16);
        const float b0 = rs_step(a0, a2, 8, u8);
        const float b1 = rs_step(a1, a3, 8, u8);
        v = rs_step(b0, b1, 4, u4);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
        sidx = (u16 ? 4 : 0) + (u8 ? 2 : 0) + (u4 ? 1 : 0);
        writer = (lane & 3) == 0;
    } else {
        static_assert(STAGES == 4, "reduce-scatter is written for 4, 8 or 16 stages");
        const float a0 = rs_step(a[0], a[2], 16, u16);
        const float a1 = rs_step(a[1], a[3], 16, u16);
        v = rs_step(a0, a1, 8, u8);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
        sidx = (u16 ? 2 : 0) + (u8 ? 1 : 0);
        writer = (lane & 7) == 0;
    }
    return v;
}

}  // namespace nvfp4
