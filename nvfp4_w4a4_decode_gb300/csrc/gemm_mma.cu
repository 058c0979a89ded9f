// gemm_mma.cu -- small-M W4A4 linear with the MAC on the tensor cores
// (mma.sync m16n8k16, f16 operands, FP32 accumulation), swap-AB: weight rows
// are the MMA's 16-row side and the M <= 8 activation rows its 8 columns, so
// the tile is fully used whatever M is (the ReSET README, "Core components"
// item 2, notes that the usual M-side tile is at most 8/128 occupied at
// M <= 8; swapping the operands removes that waste).  sm_103a has no FP4
// mma.sync, so E2M1 codes are decoded in registers with the hardware E2M1x2
// -> f16x2 conversion.
//
// Exactness.  Each block scale is folded into its operand before the MMA:
// A = e2m1(qw) * dec(sw) and B = e2m1(qx) * dec(sx) are exact in FP16 (at
// most 6 significant bits, magnitudes 2^-10 .. 2688), so the tensor core sees
// the exact dequantised products and only FP32 accumulation rounds; the
// tensor scales gX * gW are applied in FP32 at the end.  Because every
// element carries its own scale, the K order inside an MMA is free, which
// lets each lane read 16 contiguous weight bytes per row.
//
// Work layout.  K is cut into 128-element ranges.  A CTA (NW warps) owns a
// K-slice of NW * R ranges; warp w takes ranges w, w + NW, ... (R of them).
// A tile is 16 weight rows.  CTAs of one thread-block cluster (one per
// K-slice) walk the same tiles -- tile c, c + C, ... for cluster c -- two
// tiles per step, and reduce through distributed shared memory in rank order.
// Without a K split the warps reduce each tile without a CTA barrier: every
// warp stores its partial, the last one to arrive sums them in warp order.
// Per (tile, range) a lane loads rows g and g+8 (g = lane / 4), bytes
// [16 t, 16 t + 16) of the range (t = lane % 4), plus the 2 matching scale
// bytes; the next two items are in flight while one is decoded.  Registers
// stay at 64 so that two 16-warp CTAs share an SM.
// The activations of the CTA's K-slice are decoded once per CTA into shared
// memory in fragment order (conflict-free 128-bit reads), then read per range.
#include <cooperative_groups.h>

#include "formats.cuh"
#include "kernels.cuh"
#include "launch_cache.cuh"

namespace cg = cooperative_groups;

namespace nvfp4 {

namespace {

constexpr int kSlots = 4;  // tile slots of the barrier-free reduction (a multiple of 2)

struct MmaParams {
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
    int ks;  // K-slice of one CTA (elements), NW * R * 128
};

// One (tile, range) item of a lane: 16 code bytes of rows g and g + 8 and
// their two block scales each.
struct Item {
    uint4 a;       // row g
    uint4 b;       // row g + 8
    uint32_t s0;   // scale bytes of row g (two bytes) ...
    uint32_t s1;   // ... and of row g + 8, each in the register its load wrote
};

__device__ __forceinline__ uint32_t ld_u16_stream(const uint8_t* p)
{
    unsigned short v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// Two E4M3 bytes (low 16 bits) -> f16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two)
{
    uint32_t r;
    asm("{\n\t.reg .b16 lo;\n\tcvt.u16.u32 lo, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
        : "=r"(r) : "r"(two));
    return r;
}

// Broadcast the low / high half of an f16x2 to both halves.
__device__ __forceinline__ uint32_t dup_lo(uint32_t h)
{
    return __byte_perm(h, 0u, 0x1010);
}
__device__ __forceinline__ uint32_t dup_hi(uint32_t h)
{
    return __byte_perm(h, 0u, 0x3232);
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One item: 8 MMAs over the 128 elements of a range.  Lane (g, t) holds
// elements [32 t, 32 t + 32) of rows g and g + 8; MMA j takes elements
// 4j .. 4j+3 of every lane's chunk, so its A fragment is bytes 2j, 2j+1 of
// the lane's code words and its B fragment the same elements of activation
// row g (read from shared memory: one 16-byte load per word, i.e. per 2 MMAs).
__device__ __forceinline__ void mma_item(float (&acc)[4], const Item& it, const uint4* bsrc,
                                         int bstride, bool has_b)
{
    const uint32_t sa = e4m3x2_to_f16x2(it.s0);
    const uint32_t sb = e4m3x2_to_f16x2(it.s1);
    const uint32_t wa[4] = {it.a.x, it.a.y, it.a.z, it.a.w};
    const uint32_t wb[4] = {it.b.x, it.b.y, it.b.z, it.b.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {  // word w: MMAs 2w, 2w+1; block w / 2 of the chunk
        const uint32_t scA = (w < 2) ? dup_lo(sa) : dup_hi(sa);
        const uint32_t scB = (w < 2) ? dup_lo(sb) : dup_hi(sb);
        uint32_t ha[4], hb[4];
        e2m1x8_to_f16(wa[w], ha);
        e2m1x8_to_f16(wb[w], hb);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            ha[q] = hmul2(ha[q], scA);
            hb[q] = hmul2(hb[q], scB);
        }
        uint4 xb = make_uint4(0u, 0u, 0u, 0u);
        if (has_b)
            xb = bsrc[w * bstride];
        mma16816(acc, ha[0], hb[0], ha[1], hb[1], xb.x, xb.y);
        mma16816(acc, ha[2], hb[2], ha[3], hb[3], xb.z, xb.w);
    }
}

template <int R, bool PDL>
__global__ void __launch_bounds__(512, 2) mma_kernel(const MmaParams prm)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ float part[2][2][128];  // this CTA's K-slice sums per tile pair (cluster exchange)
    __shared__ unsigned s_count[kSlots];  // warps that have stored their partial of a tile slot
    if (threadIdx.x < kSlots)
        s_count[threadIdx.x] = 0u;

    if constexpr (PDL)
        asm volatile("griddepcontrol.launch_dependents;");

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, NW = blockDim.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int rank = blockIdx.x, nsplit = gridDim.x;
    const int64_t cl = blockIdx.y, ncl = gridDim.y;
    const int M = prm.m;
    const int64_t n = prm.n, kh = prm.k / 2, kb = prm.k / 16;
    const int64_t kslice0 = (int64_t)rank * prm.ks;  // first K element of this CTA
    const int nranges = prm.ks / 128;                // 128-element ranges in the slice
    const int64_t ntiles = (n + 15) / 16;
    const int64_t iters = ntiles > cl ? (ntiles - 1 - cl) / ncl + 1 : 0;

    // activation fragments [nranges][4 words][4M lanes] x 16 B, then the
    // reduction buffers [2][2 tiles][NW][128] floats
    uint4* xfrag = reinterpret_cast<uint4*>(smem_raw);
    float* red = reinterpret_cast<float*>(smem_raw + (size_t)nranges * 4 * 4 * M * 16);

    // lane's bytes of item (tile it, range i): rows (cl + it * ncl) * 16 + g (+8),
    // code bytes kr/2 + 16 t, scale bytes kr/16 + 2 t, kr = kslice0 + 128 (warp + NW i)
    const int rowA0 = (int)cl * 16 + g;
    const int tile_rows = (int)ncl * 16;
    const uint8_t* pa0 = prm.wq + (int64_t)rowA0 * kh + kslice0 / 2 + 64 * warp + 16 * t;
    const uint8_t* ps0 = prm.ws + (int64_t)rowA0 * kb + kslice0 / 16 + 8 * warp + 2 * t;
    const int64_t tstep_a = (int64_t)tile_rows * kh, tstep_s = (int64_t)tile_rows * kb;
    const int64_t row8_a = 8 * kh, row8_s = 8 * kb;
    const int code_i = 64 * NW, scale_i = 8 * NW;
    const int nrows = (int)n;
    const int niters = (int)iters;

    auto issue = [&](Item& slot, int e) {
        const int it = e / R;
        const int i = e - it * R;
        const int ra = rowA0 + it * tile_rows;
        const bool live = it < niters;
        const bool oka = live && ra < nrows, okb = live && ra + 8 < nrows;
        const uint8_t* pa = pa0 + it * tstep_a + i * code_i;
        const uint8_t* ps = ps0 + it * tstep_s + i * scale_i;
        slot.a = oka ? ld_stream_u4(pa) : make_uint4(0u, 0u, 0u, 0u);
        slot.b = okb ? ld_stream_u4(pa + row8_a) : make_uint4(0u, 0u, 0u, 0u);
        // each scale stays in its own register until it is used (combining
        // the two here would stall the loop on these loads right away)
        slot.s0 = oka ? ld_u16_stream(ps) : 0u;
        slot.s1 = okb ? ld_u16_stream(ps + row8_s) : 0u;
    };
    Item ring[2];
    issue(ring[0], 0);
    issue(ring[1], 1);

    if constexpr (PDL)
        asm volatile("griddepcontrol.wait;" ::: "memory");

    // decode this CTA's activation slice into fragment order: unit u is lane
    // (g', t') of range r, word q: elements [r*128 + 32 t' + 8 q, +8) of row g',
    // scaled by their block scale
    {
        const int units = nranges * 4 * 4 * M;
        for (int u = threadIdx.x; u < units; u += blockDim.x) {
            const int l = u % (4 * M);
            const int q = (u / (4 * M)) % 4;
            const int r = u / (16 * M);
            const int gg = l >> 2, tt = l & 3;
            const int64_t e0 = kslice0 + 128 * (int64_t)r + 32 * tt + 8 * q;
            const uint32_t codes =
                __ldg(reinterpret_cast<const uint32_t*>(prm.xq + gg * kh + e0 / 2));
            const uint32_t sc = e4m3x2_to_f16x2(__ldg(prm.xs + gg * kb + e0 / 16));
            uint32_t h[4];
            e2m1x8_to_f16(codes, h);
            const uint32_t s2 = dup_lo(sc);
            xfrag[u] = make_uint4(hmul2(h[0], s2), hmul2(h[1], s2), hmul2(h[2], s2),
                                  hmul2(h[3], s2));
        }
    }
    __syncthreads();
    const float gxw = __fmul_rn(__ldg(prm.xg), __ldg(prm.wg));

    const bool has_b = g < M;
    const int bstride = 4 * M;
    if (nsplit == 1) {
        // Whole K in this CTA: no CTA-wide barrier per tile.  Each warp stores
        // its partial tile in one of kSlots slots and counts itself in; the
        // last warp to arrive adds the NW partials in warp order and writes Y.
        // Slots are reused only after the barrier every kSlots tiles, so no
        // warp can overwrite a slot that is still being summed.
        for (int base = 0; base < niters; base += 2) {
#pragma unroll
            for (int tp = 0; tp < 2; ++tp) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    const int e = (base + tp) * R + i;
                    const int slot = (tp * R + i) & 1;
                    Item cur = ring[slot];
                    issue(ring[slot], e + 2);
                    const uint4* bsrc = xfrag + (size_t)(warp + NW * i) * 4 * bstride + lane;
                    mma_item(acc, cur, bsrc, bstride, has_b);
                }
                const int it = base + tp;
                const int ts = it % kSlots;
                reinterpret_cast<float4*>(red + ((size_t)ts * NW + warp) * 128)[lane] =
                    make_float4(acc[0], acc[1], acc[2], acc[3]);
                __threadfence_block();
                unsigned arrived = 0;
                if (lane == 0)
                    arrived = atomicAdd(&s_count[ts], 1u);
                arrived = __shfl_sync(0xFFFFFFFFu, arrived, 0);
                if (arrived == (unsigned)NW - 1) {
                    __threadfence_block();
                    for (int v = lane; v < 128; v += 32) {
                        const int lv = v >> 2, j = v & 3;
                        const int row = (lv >> 2) + 8 * (j >> 1), col = 2 * (lv & 3) + (j & 1);
                        const int r = rowA0 - g + it * tile_rows + row;
                        if (col >= M || it >= niters || r >= nrows)
                            continue;
                        const float* src = red + (size_t)ts * NW * 128 + v;
                        float sum = 0.0f;
                        for (int w = 0; w < NW; ++w)
                            sum += src[(size_t)w * 128];
                        store_y(prm.y, (int64_t)col * n + r, sum * gxw);
                    }
                    if (lane == 0)
                        s_count[ts] = 0u;
                }
            }
            if ((base + 2) % kSlots == 0)
                __syncthreads();
        }
        return;
    }
    int buf = 0;
    for (int base = 0; base < niters; base += 2) {
#pragma unroll
        for (int tp = 0; tp < 2; ++tp) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const int e = (base + tp) * R + i;
                const int slot = (tp * R + i) & 1;  // base is even: the slot is static
                Item cur = ring[slot];
                issue(ring[slot], e + 2);
                const uint4* bsrc = xfrag + (size_t)(warp + NW * i) * 4 * bstride + lane;
                mma_item(acc, cur, bsrc, bstride, has_b);
            }
            float* rb = red + ((size_t)(buf * 2 + tp) * NW + warp) * 128;
            reinterpret_cast<float4*>(rb)[lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        }
        __syncthreads();
        // fixed-order sum over the NW warps; value v = lane' * 4 + j of tile tp
        if (threadIdx.x < 256) {
            const int tp = threadIdx.x >> 7, v = threadIdx.x & 127;
            const float* src = red + ((size_t)(buf * 2 + tp) * NW) * 128 + v;
            float sum = 0.0f;
            for (int w = 0; w < NW; ++w)
                sum += src[(size_t)w * 128];
            if (nsplit == 1) {
                const int lv = v >> 2, j = v & 3;
                const int row = (lv >> 2) + 8 * (j >> 1), col = 2 * (lv & 3) + (j & 1);
                const int it = base + tp;
                const int r = rowA0 - g + it * tile_rows + row;
                if (col < M && it < niters && r < nrows)
                    store_y(prm.y, (int64_t)col * n + r, sum * gxw);
            } else {
                part[buf][tp][v] = sum;
            }
        }
        if (nsplit > 1) {
            cg::cluster_group cluster = cg::this_cluster();
            cluster.sync();
            if (rank == 0 && threadIdx.x < 256) {
                const int tp = threadIdx.x >> 7, v = threadIdx.x & 127;
                float sum = part[buf][tp][v];
                for (int rk = 1; rk < nsplit; ++rk)
                    sum += cluster.map_shared_rank(&part[0][0][0], rk)[(buf * 2 + tp) * 128 + v];
                const int lv = v >> 2, j = v & 3;
                const int row = (lv >> 2) + 8 * (j >> 1), col = 2 * (lv & 3) + (j & 1);
                const int it = base + tp;
                const int r = rowA0 - g + it * tile_rows + row;
                if (col < M && it < niters && r < nrows)
                    store_y(prm.y, (int64_t)col * n + r, sum * gxw);
            }
        }
        buf ^= 1;
    }
    if (nsplit > 1)
        cg::this_cluster().sync();  // no CTA leaves while rank 0 may still read its part[]
}

struct MmaPlan {
    int nsplit, NW, R;
};

// Split of K: nsplit CTAs per cluster (<= 8), NW warps per CTA (4..16), R
// 128-element ranges per warp and tile (1, 2, 4 or 8), with the activation
// fragments of a CTA (2 * M * K / nsplit bytes) at most 48 KB so that two
// CTAs fit on an SM (96 KB, one CTA per SM, if no split allows 48 KB).
// Fewest CTAs per cluster first, then the fewest ranges per warp.
bool plan_mma(int64_t m, int64_t k, MmaPlan* out)
{
    if (k <= 0 || k % 128 != 0)
        return false;
    const int64_t T = k / 128;
    for (int pass = 0; pass < 2; ++pass)
    for (int nsplit = 1; nsplit <= 8; ++nsplit) {
        if (T % nsplit)
            continue;
        const int64_t Tc = T / nsplit;
        if (2 * m * 128 * Tc > (pass == 0 ? 48 : 96) * 1024)
            continue;
        for (int R : {1, 2, 4, 8}) {
            if (Tc % R)
                continue;
            const int64_t nw = Tc / R;
            if (nw >= 4 && nw <= 16) {
                out->nsplit = nsplit;
                out->NW = (int)nw;
                out->R = R;
                return true;
            }
        }
    }
    return false;
}

template <int R, bool PDL>
cudaError_t launch_plan(const GemmArgs& a, const MmaPlan& p)
{
    const int threads = 32 * p.NW;
    const int ks = (int)(a.k / p.nsplit);
    const size_t smem = (size_t)(ks / 128) * 4 * 4 * a.m * 16 + sizeof(float) * kSlots * p.NW * 128;
    auto kern = mma_kernel<R, PDL>;
    const int dev = current_device();
    cudaError_t e = ensure_smem_limit(kern, smem, dev);
    if (e != cudaSuccess)
        return e;
    int per_sm = 0;
    e = cached_occupancy(kern, threads, smem, 0, dev, &per_sm);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorInvalidConfiguration;
    const int64_t ntiles = (a.n + 15) / 16;
    int64_t clusters = ((int64_t)device_sm_count(dev) * per_sm) / p.nsplit;
    if (p.nsplit > 1) {
        int maxc = 0;
        if (cached_occupancy(kern, threads, smem, p.nsplit, dev, &maxc) == cudaSuccess &&
            maxc > 0 && maxc < clusters)
            clusters = maxc;
    }
    if (clusters > ntiles)
        clusters = ntiles;
    if (clusters < 1)
        clusters = 1;

    MmaParams prm = {a.xq, a.xs, a.xg, a.wq, a.ws, a.wg, a.y, a.m, a.n, a.k, ks};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.nsplit, (unsigned)clusters, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (p.nsplit > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)p.nsplit;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (PDL) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, prm);
}

}  // namespace

bool mma_supported(int64_t m, int64_t k)
{
    MmaPlan p;
    return m >= 1 && m <= 8 && plan_mma(m, k, &p);
}

cudaError_t launch_gemm_mma(const GemmArgs& a, bool pdl)
{
    MmaPlan p;
    if (!plan_mma(a.m, a.k, &p))
        return cudaErrorInvalidValue;
    switch (p.R) {
    case 1: return pdl ? launch_plan<1, true>(a, p) : launch_plan<1, false>(a, p);
    case 2: return pdl ? launch_plan<2, true>(a, p) : launch_plan<2, false>(a, p);
    case 4: return pdl ? launch_plan<4, true>(a, p) : launch_plan<4, false>(a, p);
    default: return pdl ? launch_plan<8, true>(a, p) : launch_plan<8, false>(a, p);
    }
}

}  // namespace nvfp4
