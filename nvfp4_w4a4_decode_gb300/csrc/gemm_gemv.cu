// gemm_gemv.cu -- persistent weight-streaming small-M W4A4 kernel on the
// CUDA cores: the broadcast-weight GEMV of the ReSET README ("Core
// components" item 2), for M <= 2 (the README's `gemv_max_m=2` knob marks the
// same range; at larger M the CUDA cores run out of issue slots).
//
// Work layout.  One CTA per SM slot, each owning every C-th group of P
// consecutive weight rows (C = number of CTAs), so the row count per CTA
// differs by at most one group.  Thread t owns the 32-element chunk
// c = t % G (G = K / 32 threads per row, a multiple of 32, so a warp never
// straddles two rows) of row p = t / G of a group:
//   * weights: a group is P * K/2 contiguous bytes, read by consecutive
//     threads with 128-bit loads (each byte once, no L1 allocation), plus the
//     chunk's two E4M3 scales;  the loads of the next STAGES groups are always
//     in flight (a register ring refilled as each stage is used);
//   * activations: the thread's chunk of every X row is the same for every
//     group, so it is decoded once into registers (unscaled E2M1 as f16x2) and
//     reused -- the broadcast of the M rows is from registers;
//   * MAC: per 16-block and activation row, 8 packed HFMA2 of exact E2M1
//     products (each f16 half sums 8 products, |sum| <= 288 in steps of 1/4,
//     so the block sum is exact), then one FP32 FMA with the block's scale
//     product sx * sw;
//   * reduction, every STAGES groups: a butterfly reduce-scatter across the
//     warp's lanes leaves each group of lanes with the warp's sum for one
//     stage, those go to shared memory, and one thread per output adds the
//     G / 32 warp sums of its row in a fixed order.
// Ring slots past the end (row >= n) are not loaded; their results are
// computed from whatever the slot holds and discarded, so the hot loop needs
// no zero-fill.
//
// With programmatic dependent launch the weight prefetch is issued before
// waiting on the previous kernel; X and Y are touched only after the wait.
//
// Fused form (nvfp4_linear): the prologue quantises the FP32 activations
// itself -- the CTA's threads share the 16-blocks, run the same recipe code as
// the stand-alone quantiser (so the codes are the same bytes) into shared
// memory, and read their chunks from there; CTA 0 also stores the codes.
#include "formats.cuh"
#include "kernels.cuh"
#include "launch_cache.cuh"
#include "stream_core.cuh"

namespace nvfp4 {

namespace {

// Resident CTAs per SM the launch asks for (at most what fits).  One leaves
// half of the register file free, so that the next kernel on the stream can
// become resident under programmatic dependent launch and prefetch its
// weights while this one finishes.
#ifndef NVFP4_GEMV_CTAS_PER_SM
#define NVFP4_GEMV_CTAS_PER_SM 2
#endif
constexpr int kCtasPerSm = NVFP4_GEMV_CTAS_PER_SM;

// Registers per SM the M = 1 variants with up to 512 threads (the decode
// shapes) leave free: room for one CTA of the activation quantiser (128
// threads at up to 32 registers) beside a full complement of these CTAs, so
// that under programmatic dependent launch the next linear's quantiser is
// resident, and its prefetch of X issued, before this kernel ends.  The
// per-thread cap follows: (65536 - reserve) / (threads x CTAs per SM), in the
// allocation unit of 8.  The other variants keep the whole register file
// (tighter caps spill there).
#ifndef NVFP4_GEMV_REG_RESERVE
#define NVFP4_GEMV_REG_RESERVE 4096
#endif
__host__ __device__ constexpr int gemv_reg_cap(int m, int maxt, int minb)
{
    return (65536 - (m == 1 && maxt <= 512 ? NVFP4_GEMV_REG_RESERVE : 0)) / (maxt * minb) / 8 *
                       8 > 255
               ? 255
               : (65536 - (m == 1 && maxt <= 512 ? NVFP4_GEMV_REG_RESERVE : 0)) /
                     (maxt * minb) / 8 * 8;
}

struct GemvParams {
    const uint8_t* xq;     // quantised activations (unfused) ...
    const uint8_t* xs;
    const float* x;        // ... or FP32 activations, quantised in the prologue (fused)
    uint8_t* xq_out;       // fused: where CTA 0 stores the activation codes
    uint8_t* xs_out;       //        and block scales (both may be null)
    const float* xg;
    const uint8_t* wq;
    const uint8_t* ws;
    const float* wg;
    OutY y;
    int64_t n;
    int64_t k;
    int G;  // threads per row
    int P;  // rows per group
};

template <int M, int STAGES, int MAXT, int MINB, bool PDL, bool FUSED>
__global__ void __launch_bounds__(MAXT) __maxnreg__(gemv_reg_cap(M, MAXT, MINB))
    gemv_kernel(const GemvParams prm)
{
    static_assert(STAGES == 8 || STAGES == 4, "reduce-scatter is written for 8 or 4 stages");
    extern __shared__ __align__(16) float red[];  // [2][P][STAGES][M][G/32] warp sums,
                                                  // then (fused) X codes and scales
    if constexpr (PDL)
        asm volatile("griddepcontrol.launch_dependents;");

    const int G = prm.G, P = prm.P, WPR = G >> 5;  // warps per row
    const int t = threadIdx.x;
    const int c = t % G;
    const int p = t / G;
    const int lane = t & 31, wr = c >> 5;  // warp index within the row
    const int64_t n = prm.n, kh = prm.k / 2, kb = prm.k / 16;
    const int64_t groups = (n + P - 1) / P;
    const int64_t C = gridDim.x;
    const int64_t iters = groups > (int64_t)blockIdx.x ? (groups - 1 - blockIdx.x) / C + 1 : 0;

    // group `it` of this CTA is rows (blockIdx.x + it * C) * P + [0, P): the
    // thread's weight bytes for it sit at w0 + it * wstep
    const int64_t row0 = (int64_t)blockIdx.x * P + p;
    const uint8_t* w0 = prm.wq + row0 * kh + 16 * c;
    const uint8_t* s0 = prm.ws + row0 * kb + 2 * c;
    const int64_t wstep = C * P * kh, sstep = C * P * kb;
    const int64_t last_ok = (row0 < n) ? (n - 1 - row0) / (C * P) : -1;
    const int64_t valid_iters = iters < last_ok + 1 ? iters : last_ok + 1;

    // 1. fill the ring: weights only (independent of the previous kernel)
    uint4 rw[STAGES];
    uint32_t rs[STAGES];
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
        rw[s] = make_uint4(0u, 0u, 0u, 0u);
        rs[s] = 0u;
        if (s < valid_iters) {
            rw[s] = ld_stream_u4(w0 + s * wstep);
            rs[s] = ld_u16_nc(s0 + s * sstep);
        }
    }

    // 2. activations, after the producer of X has finished
    if constexpr (PDL)
        asm volatile("griddepcontrol.wait;" ::: "memory");
    // fused form: the CTA quantises X once, cooperatively (one 16-block per
    // task, tasks spread over all threads), into shared memory after the
    // reduction buffers; CTA 0 also stores the codes and scales
    const int nb = (int)kb;
    unsigned char* xcodes = reinterpret_cast<unsigned char*>(red + 2 * (size_t)P * STAGES * M * WPR);
    unsigned char* xscales = xcodes + (size_t)M * kh;
    if constexpr (FUSED) {
        const float g = __ldg(prm.xg);
        for (int u = t; u < M * nb; u += blockDim.x) {
            const int m = u / nb, b = u - m * nb;
            float e[16];
            const float4* src = reinterpret_cast<const float4*>(prm.x + m * prm.k + 16 * b);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 f = __ldg(src + i);
                e[4 * i + 0] = f.x;
                e[4 * i + 1] = f.y;
                e[4 * i + 2] = f.z;
                e[4 * i + 3] = f.w;
            }
            uint32_t c0, c1;
            const uint32_t sc = quantize_block16(e, g, c0, c1);
            *reinterpret_cast<uint2*>(xcodes + (size_t)m * kh + 8 * b) = make_uint2(c0, c1);
            xscales[(size_t)m * nb + b] = (unsigned char)sc;
            if (blockIdx.x == 0 && prm.xq_out != nullptr) {
                *reinterpret_cast<uint2*>(prm.xq_out + m * kh + 8 * b) = make_uint2(c0, c1);
                prm.xs_out[m * kb + b] = (uint8_t)sc;
            }
        }
        __syncthreads();
    }
    uint32_t xh[M][16];
    float sx[M][2];
#pragma unroll
    for (int m = 0; m < M; ++m) {
        uint4 v;
        uint32_t sc2;
        if constexpr (FUSED) {
            v = *reinterpret_cast<const uint4*>(xcodes + (size_t)m * kh + 16 * c);
            sc2 = *reinterpret_cast<const unsigned short*>(xscales + (size_t)m * nb + 2 * c);
        } else {
            v = __ldg(reinterpret_cast<const uint4*>(prm.xq + m * kh + 16 * c));
            sc2 = __ldg(reinterpret_cast<const unsigned short*>(prm.xs + m * kb + 2 * c));
        }
        e2m1x8_to_f16(v.x, *reinterpret_cast<uint32_t(*)[4]>(&xh[m][0]));
        e2m1x8_to_f16(v.y, *reinterpret_cast<uint32_t(*)[4]>(&xh[m][4]));
        e2m1x8_to_f16(v.z, *reinterpret_cast<uint32_t(*)[4]>(&xh[m][8]));
        e2m1x8_to_f16(v.w, *reinterpret_cast<uint32_t(*)[4]>(&xh[m][12]));
        const float2 f = e4m3x2_to_float2(sc2);
        sx[m][0] = f.x;
        sx[m][1] = f.y;
    }
    const float gxw = __fmul_rn(__ldg(prm.xg), __ldg(prm.wg));

    int buf = 0;
    for (int64_t base = 0; base < iters; base += STAGES) {
        // 3. consume the ring, refilling each stage with the group STAGES ahead
        float acc[STAGES][M];
        // running addresses of the refills (one add per stage, not a
        // multiply)
        const uint8_t* wn = w0 + (base + STAGES) * wstep;
        const uint8_t* sn = s0 + (base + STAGES) * sstep;
        const int64_t left = valid_iters - (base + STAGES);  // refills still in range
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            // M = 1 with 8 stages: decode the stage first, then refill its
            // registers (refilling first needs a copy of the stage's old
            // contents); the variants tighter on registers (M = 2, 4 stages
            // for 1024-thread CTAs) refill first, which measured faster there
            uint32_t wh[16];
            float2 sw;
            if constexpr (STAGES == 8 && M == 1) {
                e2m1x8_to_f16(rw[s].x, *reinterpret_cast<uint32_t(*)[4]>(&wh[0]));
                e2m1x8_to_f16(rw[s].y, *reinterpret_cast<uint32_t(*)[4]>(&wh[4]));
                e2m1x8_to_f16(rw[s].z, *reinterpret_cast<uint32_t(*)[4]>(&wh[8]));
                e2m1x8_to_f16(rw[s].w, *reinterpret_cast<uint32_t(*)[4]>(&wh[12]));
                sw = e4m3x2_to_float2(rs[s]);
                if (s < left) {
                    rw[s] = ld_stream_u4(wn);
                    rs[s] = ld_u16_nc(sn);
                }
            } else {
                const uint4 cw = rw[s];
                const uint32_t cs = rs[s];
                if (s < left) {
                    rw[s] = ld_stream_u4(wn);
                    rs[s] = ld_u16_nc(sn);
                }
                e2m1x8_to_f16(cw.x, *reinterpret_cast<uint32_t(*)[4]>(&wh[0]));
                e2m1x8_to_f16(cw.y, *reinterpret_cast<uint32_t(*)[4]>(&wh[4]));
                e2m1x8_to_f16(cw.z, *reinterpret_cast<uint32_t(*)[4]>(&wh[8]));
                e2m1x8_to_f16(cw.w, *reinterpret_cast<uint32_t(*)[4]>(&wh[12]));
                sw = e4m3x2_to_float2(cs);
            }
            wn += wstep;
            sn += sstep;
#pragma unroll
            for (int m = 0; m < M; ++m) {
                uint32_t p0 = 0u, p1 = 0u;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    p0 = hfma2_u32(wh[j], xh[m][j], p0);
                    p1 = hfma2_u32(wh[8 + j], xh[m][8 + j], p1);
                }
                acc[s][m] = fmaf(f16x2_sum(p1), __fmul_rn(sx[m][1], sw.y),
                                 f16x2_sum(p0) * __fmul_rn(sx[m][0], sw.x));
            }
        }
        // 4. butterfly reduce-scatter over the warp: afterwards the lanes with
        //    equal bits 4..(5 - log2 STAGES) hold the warp sum of one stage
        float* rb = red + (size_t)buf * P * STAGES * M * WPR;
#pragma unroll
        for (int m = 0; m < M; ++m) {
            float v;
            int sidx;
            bool writer;
            if constexpr (STAGES == 8) {
                const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4;
                const float a0 = rs_step(acc[0][m], acc[4][m], 16, u16);
                const float a1 = rs_step(acc[1][m], acc[5][m], 16, u16);
                const float a2 = rs_step(acc[2][m], acc[6][m], 16, u16);
                const float a3 = rs_step(acc[3][m], acc[7][m], 16, u16);
                const float b0 = rs_step(a0, a2, 8, u8);
                const float b1 = rs_step(a1, a3, 8, u8);
                v = rs_step(b0, b1, 4, u4);
                sidx = (u16 ? 4 : 0) + (u8 ? 2 : 0) + (u4 ? 1 : 0);
                writer = (lane & 3) == 0;
            } else {
                const bool u16 = lane & 16, u8 = lane & 8;
                const float a0 = rs_step(acc[0][m], acc[2][m], 16, u16);
                const float a1 = rs_step(acc[1][m], acc[3][m], 16, u16);
                v = rs_step(a0, a1, 8, u8);
                v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
                sidx = (u16 ? 2 : 0) + (u8 ? 1 : 0);
                writer = (lane & 7) == 0;
            }
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
            if (writer)
                rb[((p * STAGES + sidx) * M + m) * WPR + wr] = v;
        }
        __syncthreads();
        // 5. one thread per output: fixed-order sum of the row's warp sums
        for (int o = t; o < P * STAGES * M; o += blockDim.x) {
            const int m = o % M, s = (o / M) % STAGES, pp = o / (M * STAGES);
            float sum = 0.0f;
            for (int w = 0; w < WPR; ++w)
                sum += rb[o * WPR + w];
            const int64_t it = base + s;
            const int64_t r = ((int64_t)blockIdx.x + it * C) * P + pp;
            if (it < iters && r < n)
                store_y(prm.y, m * n + r, sum * gxw);
        }
        buf ^= 1;  // the next block writes the other buffer; one barrier per block suffices
    }
}

struct Shape {
    int G, P;
};

// One 32-element chunk per thread: G = K / 32 threads per row (K a multiple of
// 1024, at most 32768), and P rows per group so that a CTA has 256..1024
// threads.
bool pick_shape(int64_t k, Shape* out)
{
    if (k <= 0 || k % 1024 != 0 || k > 32768)
        return false;
    const int g = (int)(k / 32);
    int p = 1;
    while (g * p < 256 && g * p * 2 <= 1024)
        p *= 2;
    out->G = g;
    out->P = p;
    return true;
}

template <int M, int STAGES, int MAXT, int MINB, bool PDL, bool FUSED>
cudaError_t launch_typed(const GemmArgs& a, const Shape& sh, const FusedAct* fa)
{
    const int T = sh.G * sh.P;
    size_t smem = sizeof(float) * 2 * (size_t)sh.P * STAGES * M * (sh.G / 32);
    smem = (smem + 15) / 16 * 16;
    if (FUSED)
        smem += (size_t)M * (a.k / 2 + a.k / 16);
    auto kern = gemv_kernel<M, STAGES, MAXT, MINB, PDL, FUSED>;
    const int dev = current_device();
    if (smem > 48 * 1024) {
        cudaError_t e0 = ensure_smem_limit(kern, smem, dev);
        if (e0 != cudaSuccess)
            return e0;
    }
    int per_sm = 0;
    cudaError_t e = cached_occupancy(kern, T, smem, 0, dev, &per_sm);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorInvalidConfiguration;
    if (per_sm > kCtasPerSm)
        per_sm = kCtasPerSm;
    const int64_t groups = (a.n + sh.P - 1) / sh.P;
    int64_t grid = (int64_t)device_sm_count(dev) * per_sm;
    if (grid > groups)
        grid = groups;

    GemvParams prm = {a.xq, a.xs,
                      fa ? fa->x : nullptr, fa ? fa->xq_out : nullptr, fa ? fa->xs_out : nullptr,
                      a.xg, a.wq, a.ws, a.wg, a.y, a.n, a.k, sh.G, sh.P};
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

template <int M, bool FUSED>
cudaError_t launch_m(const GemmArgs& a, const Shape& sh, bool pdl, const FusedAct* fa)
{
    // up to 512 threads: 8 stages in flight (two 256-thread CTAs per SM);
    // larger CTAs: 4 stages, one per SM (register budget)
    const int T = sh.G * sh.P;
    if (T <= 256)
        return pdl ? launch_typed<M, 8, 256, 2, true, FUSED>(a, sh, fa)
                   : launch_typed<M, 8, 256, 2, false, FUSED>(a, sh, fa);
    if (T <= 512)
        return pdl ? launch_typed<M, 8, 512, 1, true, FUSED>(a, sh, fa)
                   : launch_typed<M, 8, 512, 1, false, FUSED>(a, sh, fa);
    return pdl ? launch_typed<M, 4, 1024, 1, true, FUSED>(a, sh, fa)
               : launch_typed<M, 4, 1024, 1, false, FUSED>(a, sh, fa);
}

}  // namespace

bool gemv_supported(int64_t m, int64_t k)
{
    Shape sh;
    return m >= 1 && m <= 2 && pick_shape(k, &sh);
}

cudaError_t launch_gemm_gemv(const GemmArgs& a, bool pdl, const FusedAct* fa)
{
    Shape sh;
    if (!pick_shape(a.k, &sh))
        return cudaErrorInvalidValue;
    if (fa != nullptr) {
        switch (a.m) {
        case 1: return launch_m<1, true>(a, sh, pdl, fa);
        case 2: return launch_m<2, true>(a, sh, pdl, fa);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (a.m) {
    case 1: return launch_m<1, false>(a, sh, pdl, nullptr);
    case 2: return launch_m<2, false>(a, sh, pdl, nullptr);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace nvfp4
