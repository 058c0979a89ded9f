// gemm_gemv.cu -- persistent weight-streaming small-M W4A4 kernel on the
// CUDA cores: the broadcast-weight GEMV of the ReSET README ("Core
// components" item 2), for M <= 2 (the README's `gemv_max_m=2` knob marks the
// same range; at larger M the CUDA cores run out of issue slots).
//
// Work layout.  One CTA per SM slot, each owning every C-th group of P
// consecutive weight rows (C = number of CTAs), so the row count per CTA
// differs by at most one group.  Thread t owns CPT 32-element chunks
// (c = t % G, G = K / (32 CPT) threads per row) of row p = t / G of a group:
//   * weights: a group is P * K/2 contiguous bytes, read by consecutive
//     threads with 128-bit loads (each byte once, no L1 allocation), plus the
//     chunk's E4M3 scales;  the loads of the next D groups are always in
//     flight (a register ring of D stages, refilled as each stage is used), so
//     the stream never stops for arithmetic or reductions;
//   * activations: the thread's chunk of every X row is the same for every
//     group, so it is decoded once into registers (unscaled E2M1 as f16x2) and
//     reused -- the broadcast of the M rows is from registers;
//   * MAC: per 16-block and activation row, 8 packed HFMA2 of exact E2M1
//     products (each f16 half sums 8 products, |sum| <= 288 in steps of 1/4,
//     so the block sum is exact), then one FP32 FMA with the block's scale
//     product sx * sw;
//   * reduction: after every D groups, the per-thread row partials go to a
//     double-buffered shared array and one warp per output sums the G
//     partials in a fixed order (lane sums, then a shuffle tree).
//
// With programmatic dependent launch the weight prefetch is issued before
// waiting on the previous kernel; X and Y are touched only after the wait.
#include "formats.cuh"
#include "kernels.cuh"

namespace nvfp4 {

namespace {

// Groups in flight per thread: 8 with one chunk per thread, 4 with two (128
// weight bytes in flight per thread); 6 / 3 for M = 2, whose activation
// registers leave less room.
template <int M, int CPT>
__host__ __device__ constexpr int stages_for()
{
    return (M == 1 ? 8 : 6) / CPT;
}

template <int CPT>
struct Slot {
    uint4 w[CPT];
    uint32_t s;  // CPT * 2 scale bytes (CPT <= 2)
};

__device__ __forceinline__ uint32_t ld_u16_nc(const uint8_t* p)
{
    unsigned short v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_u32_nc(const uint8_t* p)
{
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

template <int CPT>
__device__ __forceinline__ void load_slot(Slot<CPT>& sl, const uint8_t* wrow, const uint8_t* srow,
                                          bool valid)
{
    if (valid) {
#pragma unroll
        for (int q = 0; q < CPT; ++q)
            sl.w[q] = ld_stream_u4(wrow + 16 * q);
        sl.s = (CPT == 1) ? ld_u16_nc(srow) : ld_u32_nc(srow);
    } else {
#pragma unroll
        for (int q = 0; q < CPT; ++q)
            sl.w[q] = make_uint4(0u, 0u, 0u, 0u);
        sl.s = 0u;
    }
}

struct GemvParams {
    const uint8_t* xq;
    const uint8_t* xs;
    const float* xg;
    const uint8_t* wq;
    const uint8_t* ws;
    const float* wg;
    float* y;
    int64_t n;
    int64_t k;
    int G;  // threads per row
    int P;  // rows per group
};

template <int M, int CPT, bool PDL>
__global__ void __launch_bounds__(512) gemv_kernel(const GemvParams prm)
{
    constexpr int kStages = stages_for<M, CPT>();
    extern __shared__ float red[];  // [2][kStages * P * M][G]
    if constexpr (PDL)
        asm volatile("griddepcontrol.launch_dependents;");

    const int G = prm.G, P = prm.P;
    const int t = threadIdx.x;
    const int c = t % G;
    const int p = t / G;
    const int64_t n = prm.n, k = prm.k, kh = k / 2, kb = k / 16;
    const int64_t groups = (n + P - 1) / P;
    const int64_t C = gridDim.x;
    const int64_t iters = groups > (int64_t)blockIdx.x ? (groups - 1 - blockIdx.x) / C + 1 : 0;
    const int64_t cbyte = (int64_t)(32 * CPT / 2) * c;   // chunk byte offset in a code row
    const int64_t sbyte = (int64_t)(2 * CPT) * c;        // chunk byte offset in a scale row

    // Group `it` of this CTA holds rows (blockIdx.x + it * C) * P + [0, P): the
    // thread's weight bytes for group it sit at w0 + it * wstep.
    const int64_t row0 = (int64_t)blockIdx.x * P + p;
    const uint8_t* w0 = prm.wq + row0 * kh + cbyte;
    const uint8_t* s0 = prm.ws + row0 * kb + sbyte;
    const int64_t wstep = C * P * kh, sstep = C * P * kb;
    // the last group may be partial: rows at or past n are not loaded
    const int64_t last_ok = (row0 < n) ? (n - 1 - row0) / (C * P) : -1;  // last valid it
    const int64_t valid_iters = iters < last_ok + 1 ? iters : last_ok + 1;

    // 1. fill the ring: weights only (independent of the previous kernel)
    Slot<CPT> ring[kStages];
#pragma unroll
    for (int s = 0; s < kStages; ++s)
        load_slot<CPT>(ring[s], w0 + s * wstep, s0 + s * sstep, s < valid_iters);

    // 2. activations, after the producer of X has finished
    if constexpr (PDL)
        asm volatile("griddepcontrol.wait;" ::: "memory");
    uint32_t xh[M][16 * CPT];
    float sx[M][2 * CPT];
#pragma unroll
    for (int m = 0; m < M; ++m) {
#pragma unroll
        for (int q = 0; q < CPT; ++q) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(prm.xq + m * kh + cbyte) + q);
            e2m1x8_to_f16(v.x, *reinterpret_cast<uint32_t(*)[4]>(&xh[m][16 * q + 0]));
            e2m1x8_to_f16(v.y, *reinterpret_cast<uint32_t(*)[4]>(&xh[m][16 * q + 4]));
            e2m1x8_to_f16(v.z, *reinterpret_cast<uint32_t(*)[4]>(&xh[m][16 * q + 8]));
            e2m1x8_to_f16(v.w, *reinterpret_cast<uint32_t(*)[4]>(&xh[m][16 * q + 12]));
        }
#pragma unroll
        for (int b = 0; b < 2 * CPT; ++b)
            sx[m][b] = e4m3_to_float(__ldg(prm.xs + m * kb + sbyte + b));
    }
    const float gxw = __fmul_rn(__ldg(prm.xg), __ldg(prm.wg));

    const int OUT = kStages * P * M;
    // full warps only take part in the reduction (a CTA may end in a partial warp)
    const int warp = t >> 5, lane = t & 31, nw = blockDim.x >> 5;
    int buf = 0;
    for (int64_t base = 0; base < iters; base += kStages) {
        float* rb = red + (size_t)buf * OUT * G;
        // 3. consume the ring, refilling each stage with the group kStages ahead
#pragma unroll
        for (int s = 0; s < kStages; ++s) {
            Slot<CPT> cur = ring[s];
            {
                const int64_t it = base + kStages + s;
                load_slot<CPT>(ring[s], w0 + it * wstep, s0 + it * sstep, it < valid_iters);
            }
            float acc[M];
#pragma unroll
            for (int m = 0; m < M; ++m)
                acc[m] = 0.0f;
#pragma unroll
            for (int q = 0; q < CPT; ++q) {
                uint32_t wh[16];
                e2m1x8_to_f16(cur.w[q].x, *reinterpret_cast<uint32_t(*)[4]>(&wh[0]));
                e2m1x8_to_f16(cur.w[q].y, *reinterpret_cast<uint32_t(*)[4]>(&wh[4]));
                e2m1x8_to_f16(cur.w[q].z, *reinterpret_cast<uint32_t(*)[4]>(&wh[8]));
                e2m1x8_to_f16(cur.w[q].w, *reinterpret_cast<uint32_t(*)[4]>(&wh[12]));
                const float sw0 = e4m3_to_float((cur.s >> (16 * q)) & 0xFFu);
                const float sw1 = e4m3_to_float((cur.s >> (16 * q + 8)) & 0xFFu);
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    uint32_t p0 = 0u, p1 = 0u;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        p0 = hfma2_u32(wh[j], xh[m][16 * q + j], p0);
                        p1 = hfma2_u32(wh[8 + j], xh[m][16 * q + 8 + j], p1);
                    }
                    acc[m] = fmaf(f16x2_sum(p0), __fmul_rn(sx[m][2 * q], sw0), acc[m]);
                    acc[m] = fmaf(f16x2_sum(p1), __fmul_rn(sx[m][2 * q + 1], sw1), acc[m]);
                }
            }
#pragma unroll
            for (int m = 0; m < M; ++m)
                rb[(size_t)((s * P + p) * M + m) * G + c] = acc[m];
        }
        __syncthreads();
        // 4. one warp per output: fixed-order sum of the G row partials
        for (int o = (warp < nw ? warp : OUT); o < OUT; o += nw) {
            float v = 0.0f;
            for (int q = lane; q < G; q += 32)
                v += rb[(size_t)o * G + q];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
            if (lane == 0) {
                const int m = o % M, rp = (o / M) % P, s = o / (M * P);
                const int64_t it = base + s;
                const int64_t r = ((int64_t)blockIdx.x + it * C) * P + rp;
                if (it < iters && r < n)
                    prm.y[m * n + r] = v * gxw;
            }
        }
        buf ^= 1;  // the next block writes the other buffer; one barrier per block suffices
    }
}

struct Shape {
    int G, P, CPT;
};

// Threads per row and rows per group for a K: one 32-element chunk per
// thread while a row needs at most 512 threads, else two; P rows per group
// so that a CTA has 256..512 threads.  K must be a multiple of 1024 (2048
// above 16384) and at most 32768.
bool pick_shape(int64_t k, Shape* out)
{
    if (k <= 0 || k % 1024 != 0 || k > 32768)
        return false;
    int64_t chunks = k / 32;
    int cpt = chunks <= 512 ? 1 : 2;
    if (chunks % cpt != 0)
        return false;
    int64_t g = chunks / cpt;
    int p = 1;
    while (g * p * 2 <= 512 && g * p < 256)
        p *= 2;
    out->G = (int)g;
    out->P = p;
    out->CPT = cpt;
    return true;
}

struct DevInfo {
    int sms = 0;
};

DevInfo& dev_info()
{
    static thread_local int cached_dev = -1;
    static thread_local DevInfo info;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev != cached_dev) {
        cudaDeviceGetAttribute(&info.sms, cudaDevAttrMultiProcessorCount, dev);
        cached_dev = dev;
    }
    return info;
}

template <int M, int CPT, bool PDL>
cudaError_t launch_typed(const GemmArgs& a, const Shape& sh)
{
    const int T = sh.G * sh.P;
    const size_t smem = sizeof(float) * 2 * (size_t)stages_for<M, CPT>() * sh.P * M * sh.G;
    auto kern = gemv_kernel<M, CPT, PDL>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess)
            return e;
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, T, smem);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorInvalidConfiguration;
    if (per_sm > 2)
        per_sm = 2;  // leave room for the next kernel's CTAs (dependent launch)
    const int64_t groups = (a.n + sh.P - 1) / sh.P;
    int64_t grid = (int64_t)dev_info().sms * per_sm;
    if (grid > groups)
        grid = groups;

    GemvParams prm = {a.xq, a.xs, a.xg, a.wq, a.ws, a.wg, a.y, a.n, a.k, sh.G, sh.P};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)T, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = PDL ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, prm);
}

template <int M>
cudaError_t launch_m(const GemmArgs& a, const Shape& sh, bool pdl)
{
    if (sh.CPT == 1)
        return pdl ? launch_typed<M, 1, true>(a, sh) : launch_typed<M, 1, false>(a, sh);
    return pdl ? launch_typed<M, 2, true>(a, sh) : launch_typed<M, 2, false>(a, sh);
}

}  // namespace

bool gemv_supported(int64_t m, int64_t k)
{
    Shape sh;
    return m >= 1 && m <= 2 && pick_shape(k, &sh);
}

cudaError_t launch_gemm_gemv(const GemmArgs& a, bool pdl)
{
    Shape sh;
    if (!pick_shape(a.k, &sh))
        return cudaErrorInvalidValue;
    switch (a.m) {
    case 1: return launch_m<1>(a, sh, pdl);
    case 2: return launch_m<2>(a, sh, pdl);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace nvfp4
