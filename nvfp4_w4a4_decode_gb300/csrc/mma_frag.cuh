// mma_frag.cuh -- register-level helpers of the tensor-core (mma.sync f16)
// kernels: exact E4M3 scale pairs as f16x2, half broadcasts, the packed f16
// multiply that folds a block scale into decoded E2M1 values, and the
// m16n8k16 MMA with FP32 accumulation.
#pragma once

#include <stdint.h>

namespace nvfp4 {

// Two E4M3 bytes (low 16 bits; the first byte lands in the low half) -> f16x2,
// exact (every E4M3 value is an f16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_bits(uint32_t two)
{
    uint32_t r;
    asm("{\n\t.reg .b16 lo;\n\tcvt.u16.u32 lo, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
        : "=r"(r)
        : "r"(two));
    return r;
}

// Broadcast the low / high half of an f16x2 to both halves.
__device__ __forceinline__ uint32_t f16x2_dup_lo(uint32_t h)
{
    return __byte_perm(h, 0u, 0x1010);
}
__device__ __forceinline__ uint32_t f16x2_dup_hi(uint32_t h)
{
    return __byte_perm(h, 0u, 0x3232);
}

// Packed f16 product.  With an E2M1 value (at most 2 significant bits) and an
// E4M3 scale (at most 4) every product is exact in f16 (|p| <= 2688, and the
// smallest non-zero |p| = 2^-10 is a normal f16).
__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// D += A B for one m16n8k16 tile, f16 operands, FP32 accumulators.  Lane
// (g, t) = (lane / 4, lane % 4) holds A rows g and g + 8 at k = 2t, 2t+1
// (a0, a1) and k = 2t+8, 2t+9 (a2, a3), B column g at the same k (b0, b1),
// and D rows g, g + 8 at columns 2t, 2t+1 (d0, d1 | d2, d3).
__device__ __forceinline__ void mma_m16n8k16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Read-only, no-L1-allocate 16-bit load (scale bytes of the weight stream).
__device__ __forceinline__ uint32_t ld_stream_u16(const void* p)
{
    unsigned short v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

}  // namespace nvfp4
