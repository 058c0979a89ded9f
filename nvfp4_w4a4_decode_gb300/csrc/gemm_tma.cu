// gemm_tma.cu -- small-M W4A4 linear: TMA-fed weight stream, tensor-core MAC.
//
// Same arithmetic as the register-streaming tensor-core kernel (mma.sync
// m16n8k16, f16 operands with each E4M3 block scale folded in exactly, FP32
// accumulation, swap-AB so the M <= 8 activation rows fill the MMA's 8
// columns -- the ReSET README, "Core components" item 2, counts the usual
// M-side tile as at most 8/128 occupied), but the weight bytes arrive by bulk
// asynchronous copies (cp.async.bulk) into a ring of shared-memory stages
// instead of per-thread loads.  That keeps S - 1 whole tiles (16 rows x the
// CTA's K-slice, about 36 KB each at K = 4096) in flight per SM with no
// registers held and no per-element address arithmetic, and leaves the issue
// slots to the decode and the MMAs.
//
// Per CTA: NC consumer warps and one producer warp.  Tile it of cluster c is
// weight rows (c + it * C) * 16 .. +16.  One thread of the producer warp
// copies each row's codes and scales of the CTA's K-slice into stage
// it % S and arms that stage's mbarrier with the byte count; consumers wait
// on it (bounded), warp w takes the 128-element ranges w, w + NC, ... of the
// slice (R of them), accumulates a 16x8 tile, and the CTA (or, with a K-split
// cluster, rank 0 through distributed shared memory) sums the partials in a
// fixed order.  One barrier per tile: after it the stage is refilled with the
// tile S ahead.  Shared-memory rows are padded by 64 bytes so that the
// fragment reads of rows g and g + 8 hit distinct banks.
//
// Waits are bounded: a wait that runs out of its clock budget records
// NVFP4_DEVICE_WAIT_TIMEOUT in a device status word and the CTA skips the rest
// of its work; the host reads the word with nvfp4_device_status().
#include <cooperative_groups.h>

#include <mutex>
#include <unordered_map>

#include "../../include/nvfp4.h"
#include "formats.cuh"
#include "kernels.cuh"
#include "launch_cache.cuh"

namespace cg = cooperative_groups;

namespace nvfp4 {

__device__ unsigned int g_device_status = 0u;

namespace {

struct TmaParams {
    const uint8_t* xq;
    const uint8_t* xs;
    const float* xg;
    const uint8_t* wq;
    const uint8_t* ws;
    const float* wg;
    OutY y;
    int m;
    int n;
    int64_t k;
    int ks;        // K-slice of one CTA, a multiple of 256
    int stages;    // S
    long long wait_budget;  // clock cycles a wait may take before giving up
    int tx_skew;   // test hook: extra bytes the first stage's barrier expects
};

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Two E4M3 bytes (low 16 bits) -> f16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two)
{
    uint32_t r;
    asm("{\n\t.reg .b16 lo;\n\tcvt.u16.u32 lo, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
        : "=r"(r)
        : "r"(two));
    return r;
}

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

struct Layout {
    int cstride, sstride;        // padded stage row strides (bytes)
    size_t codes, scales, frag, red, bars, total;
};

// Stage rows are padded by 64 / 16 bytes (conflict-free fragment reads) when
// each row is its own copy (K split over a cluster); with the whole K in one
// CTA a tile's rows are contiguous in memory and arrive in one copy, unpadded.
__host__ __device__ inline Layout make_layout(int ks, int m, int nc, int stages, bool contiguous)
{
    Layout L;
    L.cstride = ks / 2 + (contiguous ? 0 : 64);
    L.sstride = ks / 16 + (contiguous ? 0 : 16);
    L.codes = 0;
    L.scales = L.codes + (size_t)stages * 16 * L.cstride;
    L.frag = L.scales + (size_t)stages * 16 * L.sstride;
    L.red = L.frag + (size_t)(ks / 128) * 4 * 4 * m * 16;
    L.bars = L.red + sizeof(float) * 2 * (size_t)nc * 128;
    L.total = L.bars + 8 * (size_t)stages;
    return L;
}

template <int R, bool PDL>
__global__ void __launch_bounds__(544, 1) tma_kernel(const TmaParams prm)
{
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ volatile int s_abort;

    if constexpr (PDL)
        asm volatile("griddepcontrol.launch_dependents;");

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int NC = (blockDim.x >> 5) - 1;  // consumer warps; the last warp produces
    const int g = lane >> 2, t = lane & 3;
    const int rank = blockIdx.x, nsplit = gridDim.x;
    const int cl = blockIdx.y, ncl = gridDim.y;
    const int M = prm.m, n = prm.n, ks = prm.ks, S = prm.stages;
    const int64_t kh = prm.k / 2, kb = prm.k / 16;
    const int64_t kslice0 = (int64_t)rank * ks;
    const int ntiles = (n + 15) / 16;
    const int iters = ntiles > cl ? (ntiles - 1 - cl) / ncl + 1 : 0;
    const bool contiguous = nsplit == 1;
    const Layout L = make_layout(ks, M, NC, S, contiguous);
    const uint32_t smem0 = smem_u32(smem);
    const bool producer = (warp == NC) && lane == 0;

    // --- stage fill: rows of tile `it` into stage it % S (producer thread)
    auto fill = [&](int it) {
        const int s = it % S;
        const int row0 = (cl + it * ncl) * 16;
        const int rows = min(16, n - row0);
        const uint32_t bar = smem0 + (uint32_t)(L.bars + 8 * s);
        uint32_t bytes = (uint32_t)rows * (uint32_t)(ks / 2 + ks / 16);
        if (it == 0)
            bytes += (uint32_t)prm.tx_skew;
        mbar_expect_tx(bar, bytes);
        if (contiguous) {  // the tile's rows are one block of memory: two copies
            bulk_g2s(smem0 + (uint32_t)(L.codes + (size_t)s * 16 * L.cstride),
                     prm.wq + (int64_t)row0 * kh, (uint32_t)rows * (uint32_t)(ks / 2), bar);
            bulk_g2s(smem0 + (uint32_t)(L.scales + (size_t)s * 16 * L.sstride),
                     prm.ws + (int64_t)row0 * kb, (uint32_t)rows * (uint32_t)(ks / 16), bar);
            return;
        }
        for (int r = 0; r < rows; ++r) {
            const int64_t row = row0 + r;
            bulk_g2s(smem0 + (uint32_t)(L.codes + ((size_t)s * 16 + r) * L.cstride),
                     prm.wq + row * kh + kslice0 / 2, (uint32_t)(ks / 2), bar);
            bulk_g2s(smem0 + (uint32_t)(L.scales + ((size_t)s * 16 + r) * L.sstride),
                     prm.ws + row * kb + kslice0 / 16, (uint32_t)(ks / 16), bar);
        }
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s)
            mbar_init(smem0 + (uint32_t)(L.bars + 8 * s), 1u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_abort = 0;
    }
    __syncthreads();
    int filled = 0;  // tiles handed to the copy engine so far (producer thread)
    if (producer)
        for (; filled < S && filled < iters; ++filled)
            fill(filled);  // weights only: independent of the previous kernel

    if constexpr (PDL)
        asm volatile("griddepcontrol.wait;" ::: "memory");

    // --- activation fragments of the slice: unit u = lane (g', t') of range q,
    // word w: elements [q*128 + 32 t' + 8 w, +8) of row g', block-scaled
    uint4* frag = reinterpret_cast<uint4*>(smem + L.frag);
    {
        const int units = (ks / 128) * 4 * 4 * M;
        for (int u = threadIdx.x; u < units; u += blockDim.x) {
            const int l = u % (4 * M);
            const int w = (u / (4 * M)) % 4;
            const int q = u / (16 * M);
            const int gg = l >> 2, tt = l & 3;
            const int64_t e0 = kslice0 + 128 * (int64_t)q + 32 * tt + 8 * w;
            const uint32_t codes =
                __ldg(reinterpret_cast<const uint32_t*>(prm.xq + gg * kh + e0 / 2));
            const uint32_t sc = e4m3x2_to_f16x2(__ldg(prm.xs + gg * kb + e0 / 16));
            uint32_t h[4];
            e2m1x8_to_f16(codes, h);
            const uint32_t s2 = dup_lo(sc);
            frag[u] = make_uint4(hmul2(h[0], s2), hmul2(h[1], s2), hmul2(h[2], s2), hmul2(h[3], s2));
        }
    }
    __syncthreads();
    const float gxw = __fmul_rn(__ldg(prm.xg), __ldg(prm.wg));
    float* red = reinterpret_cast<float*>(smem + L.red);
    const bool has_b = g < M;
    const int bstride = 4 * M;

    for (int it = 0; it < iters; ++it) {
        const int s = it % S;
        const int row0 = (cl + it * ncl) * 16;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        float acc2[4] = {0.f, 0.f, 0.f, 0.f};  // second chain: MMAs alternate between the two
        if (warp < NC) {
            // wait for the stage (bounded by the clock budget)
            const uint32_t bar = smem0 + (uint32_t)(L.bars + 8 * s);
            const uint32_t parity = (uint32_t)((it / S) & 1);
            bool ok = !s_abort;
            if (ok && !mbar_try_wait(bar, parity)) {
                const long long t0 = clock64();
                while (!(ok = mbar_try_wait(bar, parity))) {
                    if (s_abort || clock64() - t0 > prm.wait_budget) {
                        s_abort = 1;
                        atomicOr(&g_device_status, (unsigned)NVFP4_DEVICE_WAIT_TIMEOUT);
                        break;
                    }
                }
            }
            if (ok) {
                const bool va = row0 + g < n, vb = row0 + g + 8 < n;
                const unsigned char* cs = smem + L.codes + (size_t)s * 16 * L.cstride;
                const unsigned char* ss = smem + L.scales + (size_t)s * 16 * L.sstride;
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    const int q = warp + NC * i;
                    uint4 wa = make_uint4(0u, 0u, 0u, 0u), wb = wa;
                    uint32_t sa = 0u, sb = 0u;
                    if (va) {
                        wa = *reinterpret_cast<const uint4*>(cs + g * L.cstride + q * 64 + 16 * t);
                        sa = *reinterpret_cast<const unsigned short*>(ss + g * L.sstride + q * 8 + 2 * t);
                    }
                    if (vb) {
                        wb = *reinterpret_cast<const uint4*>(cs + (g + 8) * L.cstride + q * 64 + 16 * t);
                        sb = *reinterpret_cast<const unsigned short*>(ss + (g + 8) * L.sstride + q * 8 + 2 * t);
                    }
                    const uint32_t fa = e4m3x2_to_f16x2(sa), fb = e4m3x2_to_f16x2(sb);
                    const uint32_t wA[4] = {wa.x, wa.y, wa.z, wa.w};
                    const uint32_t wB[4] = {wb.x, wb.y, wb.z, wb.w};
                    const uint4* bsrc = frag + (size_t)q * 4 * bstride + lane;
#pragma unroll
                    for (int w = 0; w < 4; ++w) {  // word w: MMAs 2w, 2w+1; block w / 2
                        const uint32_t scA = (w < 2) ? dup_lo(fa) : dup_hi(fa);
                        const uint32_t scB = (w < 2) ? dup_lo(fb) : dup_hi(fb);
                        uint32_t ha[4], hb[4];
                        e2m1x8_to_f16(wA[w], ha);
                        e2m1x8_to_f16(wB[w], hb);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            ha[j] = hmul2(ha[j], scA);
                            hb[j] = hmul2(hb[j], scB);
                        }
                        uint4 xb = make_uint4(0u, 0u, 0u, 0u);
                        if (has_b)
                            xb = bsrc[w * bstride];
                        mma16816(acc, ha[0], hb[0], ha[1], hb[1], xb.x, xb.y);
                        mma16816(acc2, ha[2], hb[2], ha[3], hb[3], xb.z, xb.w);
                    }
                }
            }
            reinterpret_cast<float4*>(red + ((size_t)(it & 1) * NC + warp) * 128)[lane] =
                make_float4(acc[0] + acc2[0], acc[1] + acc2[1], acc[2] + acc2[2], acc[3] + acc2[3]);
        }
        // one barrier per tile: stage s is free, red[it & 1] is complete
        if (nsplit > 1)
            cg::this_cluster().sync();
        else
            __syncthreads();
        if (producer && it + S < iters && !s_abort) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            fill(it + S);
            filled = it + S + 1;
        }
        // fixed-order sum: ranks (rank 0 reads the others' partials), then warps
        if (threadIdx.x < 128 && (nsplit == 1 || rank == 0)) {
            const int v = threadIdx.x;
            float sum = 0.0f;
            for (int rk = 0; rk < nsplit; ++rk) {
                const float* src = red + (size_t)(it & 1) * NC * 128 + v;
                if (rk > 0)
                    src = cg::this_cluster().map_shared_rank(src, rk);
                for (int w = 0; w < NC; ++w)
                    sum += src[(size_t)w * 128];
            }
            const int lv = v >> 2, j = v & 3;
            const int row = (lv >> 2) + 8 * (j >> 1), col = 2 * (lv & 3) + (j & 1);
            const int r = row0 + row;
            if (col < M && r < n && !s_abort)
                store_y(prm.y, (int64_t)col * n + r, sum * gxw);
        }
    }
    if (nsplit > 1)
        cg::this_cluster().sync();  // no CTA leaves while rank 0 may still read its partials
    // Drain: before the CTA leaves, every copy it started has landed (waits
    // are bounded, so a stage whose barrier can never complete is given up).
    if (producer) {
        for (int st = 0; st < S && st < filled; ++st) {
            const int last = st + S * ((filled - 1 - st) / S);
            const uint32_t bar = smem0 + (uint32_t)(L.bars + 8 * st);
            const uint32_t parity = (uint32_t)((last / S) & 1);
            const long long t0 = clock64();
            while (!mbar_try_wait(bar, parity))
                if (clock64() - t0 > prm.wait_budget) {
                    atomicOr(&g_device_status, (unsigned)NVFP4_DEVICE_WAIT_TIMEOUT);
                    break;
                }
        }
    }
}

struct TmaPlan {
    int nsplit, NC, R, S, ks;
};

constexpr size_t kSmemBudget = 220 * 1024;

// K-split (cluster size <= 8, each slice a multiple of 256), NC consumer
// warps (4..16) x R 128-element ranges per warp, and the deepest ring (2..4
// stages) that fits the shared-memory budget.  Fewest ranks first; a plan with
// at least 3 stages is preferred.
bool plan_tma(int64_t m, int64_t k, TmaPlan* out)
{
    if (m < 1 || m > 8 || k <= 0 || k % 256 != 0 || k / 256 > 1 << 20)
        return false;
    for (int min_stages = 3; min_stages >= 2; --min_stages) {
        for (int nsplit = 1; nsplit <= 8; ++nsplit) {
            if (k % (256 * nsplit))
                continue;
            const int ks = (int)(k / nsplit);
            const int ranges = ks / 128;
            for (int R : {1, 2, 4, 8}) {
                if (ranges % R)
                    continue;
                const int nc = ranges / R;
                if (nc < 4 || nc > 16)
                    continue;
                int S = 0;
                for (int s = 4; s >= min_stages; --s)
                    if (make_layout(ks, (int)m, nc, s, nsplit == 1).total <= kSmemBudget) {
                        S = s;
                        break;
                    }
                if (!S)
                    continue;
                *out = {nsplit, nc, R, S, ks};
                return true;
            }
        }
    }
    return false;
}

template <int R, bool PDL>
cudaError_t launch_tma_t(const GemmArgs& a, const TmaPlan& p, long long budget, int skew)
{
    const int threads = 32 * (p.NC + 1);
    const Layout L = make_layout(p.ks, a.m, p.NC, p.S, p.nsplit == 1);
    auto kern = tma_kernel<R, PDL>;
    const int dev = current_device();
    cudaError_t e = ensure_smem_limit(kern, L.total, dev);
    if (e != cudaSuccess)
        return e;
    const int ntiles = (int)((a.n + 15) / 16);
    int clusters = device_sm_count(dev) / p.nsplit;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (p.nsplit > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)p.nsplit;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
        int maxc = 0;
        if (cached_occupancy(kern, threads, L.total, p.nsplit, dev, &maxc) == cudaSuccess &&
            maxc > 0 && maxc < clusters)
            clusters = maxc;
    }
    if (clusters > ntiles)
        clusters = ntiles;
    if (clusters < 1)
        clusters = 1;
    if (PDL) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    TmaParams prm = {a.xq, a.xs, a.xg, a.wq, a.ws, a.wg, a.y, a.m, (int)a.n, a.k,
                     p.ks, p.S, budget, skew};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.nsplit, (unsigned)clusters, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, prm);
}

}  // namespace

bool tma_supported(int64_t m, int64_t n, int64_t k)
{
    TmaPlan p;
    return n < (int64_t)1 << 30 && plan_tma(m, k, &p);
}

bool tma_single_cta_k(int64_t m, int64_t k)
{
    TmaPlan p;
    return plan_tma(m, k, &p) && p.nsplit == 1;
}

cudaError_t launch_gemm_tma(const GemmArgs& a, bool pdl, bool test_timeout)
{
    TmaPlan p;
    if (!plan_tma(a.m, a.k, &p))
        return cudaErrorInvalidValue;
    // about one second at GB300 clocks; the timeout test uses a few microseconds
    const long long budget = test_timeout ? 20000LL : 2000000000LL;
    const int skew = test_timeout ? 16 : 0;
    switch (p.R) {
    case 1: return pdl ? launch_tma_t<1, true>(a, p, budget, skew) : launch_tma_t<1, false>(a, p, budget, skew);
    case 2: return pdl ? launch_tma_t<2, true>(a, p, budget, skew) : launch_tma_t<2, false>(a, p, budget, skew);
    case 4: return pdl ? launch_tma_t<4, true>(a, p, budget, skew) : launch_tma_t<4, false>(a, p, budget, skew);
    default: return pdl ? launch_tma_t<8, true>(a, p, budget, skew) : launch_tma_t<8, false>(a, p, budget, skew);
    }
}

cudaError_t device_status_address(unsigned** out)
{
    // looked up once per device (the address of a module variable is fixed
    // for the life of the context)
    static std::mutex mu;
    static std::unordered_map<int, unsigned*> addr;
    const int dev = current_device();
    std::lock_guard<std::mutex> lock(mu);
    auto it = addr.find(dev);
    if (it != addr.end()) {
        *out = it->second;
        return cudaSuccess;
    }
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_device_status);
    if (e != cudaSuccess)
        return e;
    addr[dev] = static_cast<unsigned*>(p);
    *out = addr[dev];
    return cudaSuccess;
}

cudaError_t read_device_status(cudaStream_t stream, unsigned* out, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_device_status, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess)
        return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess || !clear)
        return e;
    const unsigned zero = 0u;
    e = cudaMemcpyToSymbolAsync(g_device_status, &zero, sizeof(unsigned), 0,
                                cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess)
        return e;
    return cudaStreamSynchronize(stream);
}

}  // namespace nvfp4
