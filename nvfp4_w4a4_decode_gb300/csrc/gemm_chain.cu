// gemm_chain.cu -- a list of independent small-M W4A4 linears in one
// persistent launch (and their activation quantisation in one launch before
// it).  The decode step of the ReSET README ("Core components" item 2; the
// trace figure runs decode at batch 1 under CUDA graphs) is a long sequence of
// such linears; launched one by one, every linear pays a launch, a ramp-up of
// its weight stream and a tail in which the last CTAs finish alone -- a few
// microseconds each, against 1.4 to 8 us of DRAM time for the 8B-shaped
// linears.  Here the weight stream never stops between linears.
//
// Work.  Linear l is cut into groups of P_l consecutive weight rows, as in the
// single-linear CUDA-core stream (gemm_gemv.cu): thread t of a CTA of T
// threads owns the 32-element chunk c = t % G_l (G_l = K_l / 32) of row
// p = t / G_l of a group, P_l = T / G_l (threads t >= P_l G_l idle for that
// linear -- whole warps, since G_l is a multiple of 32).  The groups of all
// linears are numbered one after another; CTA b owns the contiguous range
// [start[b], start[b+1]) of that list, the ranges cut so that every CTA
// streams the same number of weight bytes.  A CTA therefore crosses a handful
// of linear boundaries per launch.
//
// Stream.  Each thread keeps the loads of its next STAGES groups in flight (a
// register ring of 128-bit code loads and 16-bit scale loads, non-allocating
// in L1).  In the last block of STAGES groups of a linear the ring is
// refilled with the first groups of the CTA's next linear, so the weight
// loads do not pause at a boundary; the thread's activation chunk of the next
// linear is read (quantised codes, from L2) when its first group is consumed.
// MAC, reduction and epilogue are those of the single-linear stream: exact
// E2M1 block sums in packed FP16, one FP32 FMA per block and row with the
// block's scale product, a butterfly reduce-scatter over the warp, a
// fixed-order sum of the row's warp sums in shared memory, Y = acc * gX * gW.
// The result of every output therefore does not depend on the launch shape.
//
// The activation quantisation of all linears is one launch before the GEMM
// kernel (the same per-16-block recipe as the stand-alone quantiser, so the
// codes are the same bytes); the GEMM kernel is launched as its programmatic
// dependant: it fills its weight rings, then waits for the quantiser's codes.
#include "formats.cuh"
#include "kernels.cuh"
#include "launch_cache.cuh"
#include "stream_core.cuh"

namespace nvfp4 {

namespace {

constexpr int kMaxCtas = 512;  // CTAs of one launch (2 per SM on up to 256 SMs)

struct ChainGemmItem {
    const uint8_t* xq;
    const uint8_t* xs;
    const float* xg;
    const uint8_t* wq;
    const uint8_t* ws;
    const float* wg;
    void* y;
    int32_t n;
    int32_t k;
    int32_t G;       // threads per row, K / 32
    int32_t P;       // rows per group, T / G
    int32_t g0;      // first group of this linear in the launch's group list
    int32_t groups;  // ceil(n / P)
};

// Passed by value (kernel parameter space, read through the constant cache;
// the index is uniform across a CTA).
struct ChainGemmParams {
    int32_t count;
    int32_t y_bf16;
    int32_t start[kMaxCtas + 1];  // first group of each CTA; start[grid] = all groups
    ChainGemmItem item[kChainMaxItems];
};

struct ChainQuantItem {
    const void* x;
    const float* xg;
    uint8_t* xq;
    uint8_t* xs;
    int32_t nblocks;  // M * K / 16
    int32_t b0;       // first block of this linear in the launch's block list
};

struct ChainQuantParams {
    int32_t count;
    int32_t total;  // blocks of all linears
    ChainQuantItem item[kChainMaxItems];
};

// One CTA's share of one linear and this thread's place in it.
struct Seg {
    int item;          // index in the launch's list, -1 when there is none
    int32_t a, cnt;    // the linear's groups [a, a + cnt)
    int32_t P, c, p;   // rows per group; this thread's chunk and row in a group
    bool active;       // p < P
    int32_t valid;     // groups in [a, a + cnt) whose row p is below n
    const uint8_t* w;  // this thread's code bytes and scales in group a
    const uint8_t* s;
    int32_t wstep, sstep;  // bytes from one group to the next (P rows)
};

__device__ __forceinline__ Seg make_seg(const ChainGemmParams& prm, int i, int32_t lo, int32_t hi,
                                        int t)
{
    Seg sg;
    sg.item = -1;
    sg.cnt = 0;
    sg.valid = 0;
    if (i < 0 || i >= prm.count)
        return sg;
    const ChainGemmItem& it = prm.item[i];
    const int32_t a = lo > it.g0 ? lo - it.g0 : 0;
    const int32_t e = hi - it.g0 < it.groups ? hi - it.g0 : it.groups;
    if (e <= a)
        return sg;
    sg.item = i;
    sg.a = a;
    sg.cnt = e - a;
    sg.P = it.P;
    sg.c = t % it.G;
    sg.p = t / it.G;
    sg.active = sg.p < it.P;
    const int32_t kh = it.k / 2, kb = it.k / 16;
    const int64_t row0 = (int64_t)a * it.P + sg.p;
    sg.w = it.wq + row0 * kh + 16 * sg.c;
    sg.s = it.ws + row0 * kb + 2 * sg.c;
    sg.wstep = it.P * kh;
    sg.sstep = it.P * kb;
    if (sg.active && row0 < it.n) {
        const int32_t v = (int32_t)((it.n - row0 + it.P - 1) / it.P);
        sg.valid = v < sg.cnt ? v : sg.cnt;
    }
    return sg;
}

__host__ __device__ constexpr int chain_reg_cap(int maxt, int minb)
{
    return 65536 / (maxt * minb) / 8 * 8 > 255 ? 255 : 65536 / (maxt * minb) / 8 * 8;
}

template <int M, int STAGES, int MAXT, int MINB>
__global__ void __launch_bounds__(MAXT) __maxnreg__(chain_reg_cap(MAXT, MINB))
    gemv_chain_kernel(const __grid_constant__ ChainGemmParams prm)
{
    extern __shared__ __align__(16) float red[];  // [2][P][STAGES][M][G/32] warp sums
    asm volatile("griddepcontrol.launch_dependents;");

    const int t = threadIdx.x, lane = t & 31;
    const int32_t lo = prm.start[blockIdx.x], hi = prm.start[blockIdx.x + 1];
    if (lo >= hi)
        return;
    // the linear holding group lo (the last one whose first group is <= lo)
    int first = 0;
    {
        int b = prm.count - 1;
        while (first < b) {
            const int mid = (first + b + 1) >> 1;
            if (prm.item[mid].g0 <= lo)
                first = mid;
            else
                b = mid - 1;
        }
    }
    Seg cur = make_seg(prm, first, lo, hi, t);

    // 1. fill the ring with the first groups: weights only, before waiting
    //    for the quantised activations
    uint4 rw[STAGES];
    uint32_t rs[STAGES];
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
        rw[s] = make_uint4(0u, 0u, 0u, 0u);
        rs[s] = 0u;
        if (s < cur.valid) {
            rw[s] = ld_stream_u4(cur.w + s * cur.wstep);
            rs[s] = ld_u16_nc(cur.s + s * cur.sstep);
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");

    int buf = 0;
    while (true) {
        const ChainGemmItem& it = prm.item[cur.item];
        const int32_t n = it.n, kh = it.k / 2, kb = it.k / 16;
        const int WPR = it.G >> 5, wr = cur.c >> 5;
        XChunk<M> x;
        if (cur.active)
            load_x_chunk<M>(x, it.xq, it.xs, kh, kb, cur.c);
        const float gxw = __fmul_rn(__ldg(it.xg), __ldg(it.wg));
        const OutY y = {it.y, prm.y_bf16};
        // whether this CTA's range goes on into the next linear
        const bool more = it.g0 + cur.a + cur.cnt < hi;

        for (int32_t base = 0; base < cur.cnt; base += STAGES) {
            // in the last block the refills are the next linear's first groups
            int32_t nv = 0, nws = 0, nss = 0;
            const uint8_t *nw = nullptr, *ns = nullptr;
            if (base + STAGES >= cur.cnt && more) {
                const Seg nx = make_seg(prm, cur.item + 1, lo, hi, t);
                nv = nx.valid;
                nw = nx.w;
                ns = nx.s;
                nws = nx.wstep;
                nss = nx.sstep;
            }
            float acc[STAGES][M];
            const uint8_t* wn = cur.w + (int64_t)(base + STAGES) * cur.wstep;
            const uint8_t* sn = cur.s + (int64_t)(base + STAGES) * cur.sstep;
            const int32_t left = cur.valid - (base + STAGES);  // refills still in this linear
#pragma unroll
            for (int s = 0; s < STAGES; ++s) {
                uint32_t wh[16];
                float2 sw;
                if constexpr (STAGES >= 8 && M == 1) {
                    // decode the stage, then refill its registers
                    decode_w_chunk(rw[s], wh);
                    sw = e4m3x2_to_float2(rs[s]);
                    if (s < left) {
                        rw[s] = ld_stream_u4(wn);
                        rs[s] = ld_u16_nc(sn);
                    } else if (s < nv) {
                        rw[s] = ld_stream_u4(nw + s * nws);
                        rs[s] = ld_u16_nc(ns + s * nss);
                    }
                } else {
                    const uint4 cw = rw[s];
                    const uint32_t cs = rs[s];
                    if (s < left) {
                        rw[s] = ld_stream_u4(wn);
                        rs[s] = ld_u16_nc(sn);
                    } else if (s < nv) {
                        rw[s] = ld_stream_u4(nw + s * nws);
                        rs[s] = ld_u16_nc(ns + s * nss);
                    }
                    decode_w_chunk(cw, wh);
                    sw = e4m3x2_to_float2(cs);
                }
                wn += cur.wstep;
                sn += cur.sstep;
                mac_chunk<M>(wh, sw, x, acc[s]);
            }
            // reduce-scatter over the warp, one warp sum per (row, stage, m)
            // into shared memory; idle warps (p >= P) write nothing
            float* rb = red + (size_t)buf * STAGES * M * (blockDim.x >> 5);
            if (cur.active) {
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    float a[STAGES];
#pragma unroll
                    for (int s = 0; s < STAGES; ++s)
                        a[s] = acc[s][m];
                    int sidx;
                    bool writer;
                    const float v = reduce_scatter<STAGES>(a, lane, sidx, writer);
                    if (writer)
                        rb[((cur.p * STAGES + sidx) * M + m) * WPR + wr] = v;
                }
            }
            __syncthreads();
            // one thread per output: fixed-order sum of the row's warp sums
            for (int o = t; o < cur.P * STAGES * M; o += blockDim.x) {
                const int m = o % M, s = (o / M) % STAGES, pp = o / (M * STAGES);
                float sum = 0.0f;
                for (int w = 0; w < WPR; ++w)
                    sum += rb[o * WPR + w];
                const int64_t r = (int64_t)(cur.a + base + s) * cur.P + pp;
                if (base + s < cur.cnt && r < n)
                    store_y(y, m * (int64_t)n + r, sum * gxw);
            }
            buf ^= 1;  // the next block writes the other buffer
        }
        if (!more)
            break;
        cur = make_seg(prm, cur.item + 1, lo, hi, t);  // its first groups are in the ring
        if (cur.item < 0)
            break;
    }
}

// Activation quantisation of every linear of the launch: four threads per
// 16-element block (the quad's amax by shuffles, the E4M3 scale, each
// thread's four E2M1 codes, the two code words gathered by a shuffle), the
// blocks of all linears numbered one after another.  The loop bound is
// uniform across a warp, so every shuffle has its whole warp.
template <bool BF16>
__global__ void __launch_bounds__(128) quantize_chain_kernel(
    const __grid_constant__ ChainQuantParams prm)
{
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31, sub = lane & 3;
    const int64_t q0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 2;
    const int64_t stride = ((int64_t)gridDim.x * blockDim.x) >> 2;
    for (int64_t b = q0; b - (lane >> 2) < prm.total; b += stride) {
        const bool valid = b < prm.total;
        int i = 0;
        if (valid) {
            int hi = prm.count - 1;
            while (i < hi) {
                const int mid = (i + hi + 1) >> 1;
                if (prm.item[mid].b0 <= b)
                    i = mid;
                else
                    hi = mid - 1;
            }
        }
        const ChainQuantItem& it = prm.item[i];
        const int64_t lb = b - it.b0;  // block within this linear (row-major)
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (valid) {
            if constexpr (BF16) {
                const uint2 raw = __ldg(reinterpret_cast<const uint2*>(it.x) + 4 * lb + sub);
                v = make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                                __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u));
            } else {
                v = __ldg(reinterpret_cast<const float4*>(it.x) + 4 * lb + sub);
            }
        }
        float bmax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
        bmax = fmaxf(bmax, __shfl_xor_sync(0xFFFFFFFFu, bmax, 1));
        bmax = fmaxf(bmax, __shfl_xor_sync(0xFFFFFFFFu, bmax, 2));
        float S;
        const uint32_t sc = block_scale(bmax, valid ? __ldg(it.xg) : 0.0f, S);
        const float e[4] = {v.x, v.y, v.z, v.w};
        const BlockDivisor d = make_divisor(S);
        uint32_t codes = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            codes |= element_code_div(e[j], d) << (4 * j);
        const uint32_t mine = codes << (16 * (sub & 1));
        const uint32_t word = mine | __shfl_xor_sync(0xFFFFFFFFu, mine, 1);
        if (valid && (sub & 1) == 0)
            reinterpret_cast<uint32_t*>(it.xq)[2 * lb + (sub >> 1)] = word;
        if (valid && sub == 0)
            it.xs[lb] = (uint8_t)sc;
    }
}

// ---- host side -----------------------------------------------------------------

struct Variant {
    int maxt, minb, stages;
};

// Threads per CTA for the linears of one launch: every row must fit a CTA
// (T >= G_l); among the compiled variants the smallest that takes the widest
// row.  Up to 256 threads: two CTAs per SM with 8 groups in flight per thread;
// 384 threads (the 8B-shaped decode layers: K = 4096 and 12288 use all 384):
// one CTA with 16 in flight (8 at M = 2, for registers); up to 512: one CTA
// with 8; wider rows: one CTA of up to 1024 threads with 4 in flight.
Variant pick_variant(int m, int gmax, int* T)
{
    if (gmax <= 256) {
        *T = 256;
        return {256, 2, 8};
    }
    if (gmax <= 384) {
        *T = 384;
        return {384, 1, m == 1 ? 16 : 8};
    }
    if (gmax <= 512) {
        *T = 512;
        return {512, 1, 8};
    }
    *T = (gmax + 31) / 32 * 32;
    return {1024, 1, 4};
}

template <int M, int STAGES, int MAXT, int MINB>
cudaError_t launch_chain_gemm_t(ChainGemmParams& prm, int T, int64_t total_bytes,
                                const int64_t* item_group_bytes, cudaStream_t stream, bool pdl)
{
    auto kern = gemv_chain_kernel<M, STAGES, MAXT, MINB>;
    const int dev = current_device();
    const size_t smem = sizeof(float) * 2 * (size_t)STAGES * M * (T / 32);
    int per_sm = 0;
    cudaError_t e = cached_occupancy(kern, T, smem, 0, dev, &per_sm);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorInvalidConfiguration;
    if (per_sm > MINB)
        per_sm = MINB;
    int grid = device_sm_count(dev) * per_sm;
    const int32_t groups = prm.item[prm.count - 1].g0 + prm.item[prm.count - 1].groups;
    if (grid > kMaxCtas)
        grid = kMaxCtas;
    if (grid > groups)
        grid = groups;
    // cut the group list into `grid` ranges of (nearly) equal weight bytes
    int i = 0;
    int64_t before = 0;  // bytes of the linears before item i
    for (int b = 0; b <= grid; ++b) {
        const int64_t target = total_bytes * b / grid;
        while (i < prm.count - 1 && before + prm.item[i].groups * item_group_bytes[i] <= target) {
            before += prm.item[i].groups * item_group_bytes[i];
            ++i;
        }
        int64_t g = prm.item[i].g0 + (target - before + item_group_bytes[i] - 1) / item_group_bytes[i];
        if (g > groups)
            g = groups;
        prm.start[b] = (int32_t)g;
    }
    prm.start[0] = 0;
    prm.start[grid] = groups;
    for (int b = 1; b <= grid; ++b)  // non-decreasing, whatever the rounding
        if (prm.start[b] < prm.start[b - 1])
            prm.start[b] = prm.start[b - 1];

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)T, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, prm);
}

template <int M>
cudaError_t launch_chain_gemm_m(ChainGemmParams& prm, const Variant& v, int T, int64_t total,
                                const int64_t* gb, cudaStream_t s, bool pdl)
{
    if (v.maxt == 256)
        return launch_chain_gemm_t<M, 8, 256, 2>(prm, T, total, gb, s, pdl);
    if (v.maxt == 384)
        return launch_chain_gemm_t<M, (M == 1 ? 16 : 8), 384, 1>(prm, T, total, gb, s, pdl);
    if (v.maxt == 512)
        return launch_chain_gemm_t<M, 8, 512, 1>(prm, T, total, gb, s, pdl);
    return launch_chain_gemm_t<M, 4, 1024, 1>(prm, T, total, gb, s, pdl);
}

}  // namespace

cudaError_t launch_chain_quant(const ChainLinear* items, int count, int m, bool x_bf16,
                               cudaStream_t stream, bool pdl)
{
    ChainQuantParams prm;
    prm.count = count;
    int64_t total = 0;
    for (int i = 0; i < count; ++i) {
        prm.item[i] = {items[i].x, items[i].xg, items[i].xq, items[i].xs,
                       (int32_t)(m * items[i].k / 16), (int32_t)total};
        total += m * items[i].k / 16;
    }
    prm.total = (int32_t)total;
    const int dev = current_device();
    int64_t grid = (4 * total + 127) / 128;
    const int64_t cap = (int64_t)device_sm_count(dev) * 16;
    if (grid > cap)
        grid = cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return x_bf16 ? cudaLaunchKernelEx(&cfg, quantize_chain_kernel<true>, prm)
                  : cudaLaunchKernelEx(&cfg, quantize_chain_kernel<false>, prm);
}

bool chain_shape_ok(int64_t m, int64_t n, int64_t k)
{
    return m >= 1 && m <= 2 && n >= 1 && n < (int64_t(1) << 30) && k >= 1024 && k % 1024 == 0 &&
           k <= 32768;
}

cudaError_t launch_linear_chain(const ChainLinear* items, int count, int m, bool quantize,
                                bool x_bf16, bool y_bf16, cudaStream_t stream, bool pdl)
{
    if (count < 1 || count > kChainMaxItems || m < 1 || m > 2)
        return cudaErrorInvalidValue;
    int gmax = 0;
    for (int i = 0; i < count; ++i)
        if (items[i].k / 32 > gmax)
            gmax = (int)(items[i].k / 32);
    int T = 0;
    const Variant v = pick_variant(m, gmax, &T);
    ChainGemmParams prm;
    prm.count = count;
    prm.y_bf16 = y_bf16 ? 1 : 0;
    int64_t gb[kChainMaxItems];
    int64_t total = 0, groups = 0;
    for (int i = 0; i < count; ++i) {
        const ChainLinear& L = items[i];
        const int32_t G = (int32_t)(L.k / 32), P = T / G;
        const int32_t ng = (int32_t)((L.n + P - 1) / P);
        prm.item[i] = {L.xq, L.xs, L.xg, L.wq, L.ws, L.wg, L.y, (int32_t)L.n, (int32_t)L.k,
                       G, P, (int32_t)groups, ng};
        gb[i] = (int64_t)P * L.k * 9 / 16;  // weight bytes of a group
        total += ng * gb[i];
        groups += ng;
    }
    if (groups >= (int64_t(1) << 31))
        return cudaErrorInvalidValue;
    bool gemm_pdl = pdl;
    if (quantize) {
        const cudaError_t e = launch_chain_quant(items, count, m, x_bf16, stream, pdl);
        if (e != cudaSuccess)
            return e;
        gemm_pdl = true;  // the GEMM's weight prefetch does not depend on the quantiser
    }
    return m == 1 ? launch_chain_gemm_m<1>(prm, v, T, total, gb, stream, gemm_pdl)
                  : launch_chain_gemm_m<2>(prm, v, T, total, gb, stream, gemm_pdl);
}

}  // namespace nvfp4
