// gemm_gemv.cu -- weight-streaming small-M W4A4 kernel on the CUDA cores
// (the broadcast-weight GEMV of the ReSET README, "Core components" item 2,
// for M <= 2: the README's `gemv_max_m=2` knob marks the same range).
//
// Layout of the work.  A CTA owns a tile of RT consecutive weight rows and a
// K-slice of KS columns; the K-slices of one tile form a thread-block cluster
// of K/KS CTAs that reduce through distributed shared memory.  Inside the
// CTA, thread t owns the 32-element chunk c = t % G (G = KS/32) of the slice
// and walks the rows p, p + P, p + 2P, ... (p = t / G), so:
//   * weights: each row pass of P rows is P * KS/2 contiguous bytes read by
//     consecutive threads with one 128-bit load each (fully coalesced, each
//     byte read once, no L1 allocation), plus one 16-bit load of the chunk's
//     two E4M3 scales;
//   * activations: the thread's chunk of every X row is fixed, so it is
//     decoded once into registers (unscaled E2M1 as f16x2) and reused for
//     all RT/P rows -- the "broadcast" is from registers, not shared memory;
//   * MAC: per 16-block and activation row, 8 packed HFMA2 of exact E2M1
//     products (each f16 half sums 8 products, |sum| <= 288 in steps of 1/4:
//     exact), then one FP32 FMA with the block's scale product sx * sw;
//   * reduction: per-thread row partials go through shared memory and are
//     summed in a fixed order by one warp per output (lane partial sums, then
//     a warp-shuffle tree), then across the cluster in rank order.
// All loads of a CTA are issued before any arithmetic, which keeps
// RT/P * 18 bytes per thread in flight.
#include <cooperative_groups.h>

#include "formats.cuh"
#include "kernels.cuh"

namespace cg = cooperative_groups;

namespace nvfp4 {

namespace {

template <int M, int KS, int P, int PASSES>
struct GemvCfg {
    static constexpr int G = KS / 32;        // threads per row (one chunk each)
    static constexpr int T = G * P;          // threads per CTA
    static constexpr int RT = P * PASSES;    // rows per tile
    static constexpr int OUT = RT * M;       // outputs per tile
    static_assert(G % 32 == 0, "a warp must stay inside one row");
    static constexpr size_t smem_bytes = sizeof(float) * (size_t)OUT * G + sizeof(float) * OUT;
};

__device__ __forceinline__ uint32_t ld_u16_nc(const uint8_t* p)
{
    unsigned short v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

template <int M, int KS, int P, int PASSES, bool PDL>
__global__ void __launch_bounds__(GemvCfg<M, KS, P, PASSES>::T)
gemv_kernel(const uint8_t* __restrict__ xq, const uint8_t* __restrict__ xs,
            const float* __restrict__ xg, const uint8_t* __restrict__ wq,
            const uint8_t* __restrict__ ws, const float* __restrict__ wg,
            float* __restrict__ y, int64_t n, int64_t k)
{
    using C = GemvCfg<M, KS, P, PASSES>;
    extern __shared__ float smem[];
    float* red = smem;                      // [OUT][G]
    float* part = smem + (size_t)C::OUT * C::G;  // [OUT], this CTA's slice sums

    const int t = threadIdx.x;
    const int c = t % C::G;
    const int p = t / C::G;
    const int kslice = blockIdx.y;
    const int64_t row0 = (int64_t)blockIdx.x * C::RT;
    const int64_t kh = k / 2, kb = k / 16;
    const int64_t cbyte = (int64_t)kslice * (KS / 2) + 16 * c;
    const int64_t sbyte = (int64_t)kslice * (KS / 16) + 2 * c;

    // 1. weight stream: every load of the tile in flight at once
    uint4 wv[PASSES];
    uint32_t sv[PASSES];
#pragma unroll
    for (int i = 0; i < PASSES; ++i) {
        const int64_t r = row0 + (int64_t)i * P + p;
        if (r < n) {
            wv[i] = ld_stream_u4(wq + r * kh + cbyte);
            sv[i] = ld_u16_nc(ws + r * kb + sbyte);
        } else {
            wv[i] = make_uint4(0u, 0u, 0u, 0u);
            sv[i] = 0u;
        }
    }

    // 2. activations (written by the preceding quantiser: wait for it first
    //    when launched as a programmatic dependent)
    if constexpr (PDL)
        asm volatile("griddepcontrol.wait;" ::: "memory");
    uint32_t xh[M][16];
    float sx[M][2];
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(xq + m * kh + cbyte));
        const uint32_t s = __ldg(reinterpret_cast<const unsigned short*>(xs + m * kb + sbyte));
        e2m1x8_to_f16(v.x, *reinterpret_cast<uint32_t(*)[4]>(&xh[m][0]));
        e2m1x8_to_f16(v.y, *reinterpret_cast<uint32_t(*)[4]>(&xh[m][4]));
        e2m1x8_to_f16(v.z, *reinterpret_cast<uint32_t(*)[4]>(&xh[m][8]));
        e2m1x8_to_f16(v.w, *reinterpret_cast<uint32_t(*)[4]>(&xh[m][12]));
        sx[m][0] = e4m3_to_float(s & 0xFFu);
        sx[m][1] = e4m3_to_float(s >> 8);
    }

    // 3. decode each weight chunk once, broadcast it over the M rows
    float acc[PASSES][M];
#pragma unroll
    for (int i = 0; i < PASSES; ++i) {
        uint32_t wh[16];
        e2m1x8_to_f16(wv[i].x, *reinterpret_cast<uint32_t(*)[4]>(&wh[0]));
        e2m1x8_to_f16(wv[i].y, *reinterpret_cast<uint32_t(*)[4]>(&wh[4]));
        e2m1x8_to_f16(wv[i].z, *reinterpret_cast<uint32_t(*)[4]>(&wh[8]));
        e2m1x8_to_f16(wv[i].w, *reinterpret_cast<uint32_t(*)[4]>(&wh[12]));
        const float sw0 = e4m3_to_float(sv[i] & 0xFFu);
        const float sw1 = e4m3_to_float(sv[i] >> 8);
#pragma unroll
        for (int m = 0; m < M; ++m) {
            uint32_t p0 = 0u, p1 = 0u;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                p0 = hfma2_u32(wh[j], xh[m][j], p0);
                p1 = hfma2_u32(wh[8 + j], xh[m][8 + j], p1);
            }
            acc[i][m] = fmaf(f16x2_sum(p1), __fmul_rn(sx[m][1], sw1),
                             f16x2_sum(p0) * __fmul_rn(sx[m][0], sw0));
        }
    }

    // 4. reduce over the G threads of each row, fixed order
#pragma unroll
    for (int i = 0; i < PASSES; ++i)
#pragma unroll
        for (int m = 0; m < M; ++m)
            red[(size_t)((i * P + p) * M + m) * C::G + c] = acc[i][m];
    __syncthreads();
    const int warp = t >> 5, lane = t & 31;
    constexpr int NW = C::T / 32;
    for (int o = warp; o < C::OUT; o += NW) {
        float v = 0.0f;
#pragma unroll
        for (int q = 0; q < C::G / 32; ++q)
            v += red[(size_t)o * C::G + q * 32 + lane];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
        if (lane == 0)
            part[o] = v;
    }

    // 5. across the K-slices of the cluster (rank order), then the epilogue
    const float gxw = __fmul_rn(__ldg(xg), __ldg(wg));
    if (gridDim.y == 1) {
        __syncthreads();
        for (int o = t; o < C::OUT; o += C::T) {
            const int rt = o / M, m = o % M;
            const int64_t r = row0 + rt;
            if (r < n)
                y[m * n + r] = part[o] * gxw;
        }
        return;
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    if (kslice == 0) {
        const int ranks = (int)gridDim.y;
        for (int o = t; o < C::OUT; o += C::T) {
            float v = part[o];
            for (int rk = 1; rk < ranks; ++rk)
                v += cluster.map_shared_rank(part, rk)[o];
            const int rt = o / M, m = o % M;
            const int64_t r = row0 + rt;
            if (r < n)
                y[m * n + r] = v * gxw;
        }
    }
    cluster.sync();  // keep every slice's shared memory alive until read
}

template <int M, int KS, int P, int PASSES>
cudaError_t launch_cfg(const GemmArgs& a, int ksplit, bool pdl)
{
    using C = GemvCfg<M, KS, P, PASSES>;
    const size_t smem = C::smem_bytes;
    auto kern = pdl ? gemv_kernel<M, KS, P, PASSES, true> : gemv_kernel<M, KS, P, PASSES, false>;
    static bool configured[2] = {false, false};
    if (!configured[pdl]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess)
            return e;
        configured[pdl] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.n + C::RT - 1) / C::RT), (unsigned)ksplit, 1);
    cfg.blockDim = dim3(C::T, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = (unsigned)ksplit;
    attr[na].val.clusterDim.z = 1;
    ++na;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, a.xq, a.xs, a.xg, a.wq, a.ws, a.wg, a.y, a.n, a.k);
}

template <int M>
cudaError_t launch_m(const GemmArgs& a, int ks, bool pdl)
{
    const int ksplit = (int)(a.k / ks);
    switch (ks) {
    case 2048: return launch_cfg<M, 2048, 4, 8>(a, ksplit, pdl);
    case 4096: return launch_cfg<M, 4096, 2, 8>(a, ksplit, pdl);
    case 5120: return launch_cfg<M, 5120, 2, 8>(a, ksplit, pdl);
    case 6144: return launch_cfg<M, 6144, 1, 8>(a, ksplit, pdl);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

// K-slice for the CUDA-core kernel: the largest supported slice that divides
// K into at most 8 cluster ranks (0 if none does).
int gemv_pick_slice(int64_t k)
{
    static const int cand[] = {4096, 5120, 6144, 2048};
    for (int ks : cand)
        if (k % ks == 0 && k / ks <= 8)
            return ks;
    return 0;
}

cudaError_t launch_gemm_gemv(const GemmArgs& a, int ks, bool pdl)
{
    switch (a.m) {
    case 1: return launch_m<1>(a, ks, pdl);
    case 2: return launch_m<2>(a, ks, pdl);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace nvfp4
