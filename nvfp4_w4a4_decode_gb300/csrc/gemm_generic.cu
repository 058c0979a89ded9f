// gemm_generic.cu -- the shape-general small-M W4A4 kernel (CUDA cores).
//
// Y[m][n] = gX gW sum_b sx[m][b] sw[n][b] sum_{i in b} qx[m][i] qw[n][i] for
// any K that is a multiple of 16: the broadcast-weight GEMV of the ReSET
// README ("Core components" item 2) in its plainest form.  One warp per
// output row n; lane l takes the 16-element blocks b = l, l + 32, ...; each
// weight block is decoded once and reused for all M activation rows.
//
// Exactness of the inner sum: E2M1 products are multiples of 1/4 of
// magnitude <= 36, and each half of an f16x2 accumulator sums 8 of them
// (<= 288 = 1152 quarters < 2^11), so the per-block sum is exact in FP16 and
// in FP32 after conversion; only the FP32 accumulation across blocks rounds.
#include "formats.cuh"
#include "kernels.cuh"

namespace nvfp4 {

template <int M>
__global__ void __launch_bounds__(256) gemm_generic_kernel(
    const uint8_t* __restrict__ xq, const uint8_t* __restrict__ xs, const float* __restrict__ xg,
    const uint8_t* __restrict__ wq, const uint8_t* __restrict__ ws, const float* __restrict__ wg,
    const OutY y, int64_t n, int64_t k)
{
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (row >= n)
        return;
    const int64_t kh = k / 2, kb = k / 16;
    const uint8_t* wrow = wq + row * kh;
    const uint8_t* srow = ws + row * kb;

    float acc[M];
#pragma unroll
    for (int m = 0; m < M; ++m)
        acc[m] = 0.0f;

    for (int64_t b = lane; b < kb; b += 32) {
        const uint2 wv = ld_stream_u2(wrow + 8 * b);
        const float sw = e4m3_to_float(__ldg(srow + b));
        uint32_t wh[8];
        e2m1x8_to_f16(wv.x, *reinterpret_cast<uint32_t(*)[4]>(&wh[0]));
        e2m1x8_to_f16(wv.y, *reinterpret_cast<uint32_t(*)[4]>(&wh[4]));
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const uint2 xv = __ldg(reinterpret_cast<const uint2*>(xq + m * kh) + b);
            const float sx = e4m3_to_float(__ldg(xs + m * kb + b));
            uint32_t xh[8];
            e2m1x8_to_f16(xv.x, *reinterpret_cast<uint32_t(*)[4]>(&xh[0]));
            e2m1x8_to_f16(xv.y, *reinterpret_cast<uint32_t(*)[4]>(&xh[4]));
            uint32_t p = 0u;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                p = hfma2_u32(wh[i], xh[i], p);
            acc[m] = fmaf(f16x2_sum(p), __fmul_rn(sx, sw), acc[m]);
        }
    }

#pragma unroll
    for (int m = 0; m < M; ++m) {
        float v = acc[m];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
        acc[m] = v;
    }
    if (lane == 0) {
        const float gxw = __fmul_rn(__ldg(xg), __ldg(wg));
#pragma unroll
        for (int m = 0; m < M; ++m)
            store_y(y, m * n + row, acc[m] * gxw);
    }
}

template <int M>
static cudaError_t launch_generic_m(const GemmArgs& a)
{
    const int64_t grid = (a.n + 7) / 8;
    gemm_generic_kernel<M><<<(unsigned)grid, 256, 0, a.stream>>>(a.xq, a.xs, a.xg, a.wq, a.ws,
                                                                 a.wg, a.y, a.n, a.k);
    return cudaGetLastError();
}

cudaError_t launch_gemm_generic(const GemmArgs& a)
{
    switch (a.m) {
    case 1: return launch_generic_m<1>(a);
    case 2: return launch_generic_m<2>(a);
    case 3: return launch_generic_m<3>(a);
    case 4: return launch_generic_m<4>(a);
    case 5: return launch_generic_m<5>(a);
    case 6: return launch_generic_m<6>(a);
    case 7: return launch_generic_m<7>(a);
    case 8: return launch_generic_m<8>(a);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace nvfp4
