// gemm_splitk.cu -- small-M W4A4 linear on the tensor cores, K split into
// chunks and every warp streaming its own work items (mma.sync m16n8k16, f16
// operands, FP32 accumulation, swap-AB: weight rows are the MMA's 16-row side
// and the M <= 8 activation rows its 8 columns).  Used for the whole M <= 8
// range: the ReSET README ("Core components" item 2) streams the weights past
// the activations for decode; this kernel keeps that pattern (each weight
// byte read once, activations resident on chip) and moves the MAC onto the
// tensor cores.
//
// Exactness.  Every 16-block scale is folded into its operand before the MMA
// (e2m1 * dec(scale) is exact in f16), so the tensor core sees the exact
// dequantised products and only FP32 accumulation rounds; gX * gW is applied
// at the end.  Because each element carries its own scale, the order of K
// inside an MMA is free: each lane takes the bytes that make its loads whole
// 32-byte sectors.
//
// Work layout.  K is cut into nch chunks of whole 256-element sub-items, as
// equal as they can be: the first r = (K / 256) % nch chunks one sub-item
// longer than the others (at most kc elements, kc <= 32768 / M).  CTA (c, y)
// of the (nch, Cy) grid -- one 16-warp CTA per SM -- owns chunk c.  Its warps form groups of grp warps (1, 2, 4, 8 or
// 16); group gi owns the tiles (16 weight rows) y * ngrp + gi + j * Cy * ngrp,
// and warp r of the group takes the sub-items (256 elements of K) r, r + grp,
// ... of each tile's chunk.  After the prologue a warp streams its sub-items
// through its own ring of kStages shared-memory slots filled by cp.async
// (every lane copies its own 16-byte pieces; the quad copies a row's scale
// bytes, so a warp barrier follows each wait), accumulates a tile's 16 x 8
// block in registers and, at the end of its share of the tile,
//   * adds the group's partials (shared memory, one named barrier per tile,
//     rank order) in rank 0, which then
//   * writes Y directly when K is one chunk, or
//   * stores the partial in the workspace and counts it in; the warp that
//     stores a tile's last partial sums all of them in chunk order (so the
//     result does not depend on which warp finishes last), writes Y and
//     resets the tile's counter to zero for the next call; or
//   * (cluster form: where the planner finds it cheaper, and for calls
//     without the workspace a split needs) keeps the partial in its own
//     shared memory: the nch CTAs of one tile set form a thread-block
//     cluster (chunk = rank), and after the stream every warp of the cluster
//     sums some of the set's tiles, reading the nch partials through
//     distributed shared memory in chunk order, and writes Y.
// There is no CTA-wide barrier after the prologue and no wait on another CTA
// (the cluster form's two cluster barriers at the end aside).
// Per sub-item, lane (g, t) = (lane / 4, lane % 4) copies of rows g and g + 8
// the code bytes [16t, 16t + 16) and [64 + 16t, 64 + 16t + 16) of the row's
// 128 (so one copy instruction covers two whole sectors per row) and uses the
// scale bytes {2t, 2t + 1} and {8 + 2t, 9 + 2t}.
// The activations of the chunk are decoded once per CTA, scaled, into shared
// memory in fragment order (one conflict-free 16-byte read per two MMAs), for
// the M real columns only.
#include <cooperative_groups.h>

#include <mutex>
#include <unordered_map>

#include "formats.cuh"
#include "kernels.cuh"
#include "launch_cache.cuh"
#include "mma_frag.cuh"

namespace nvfp4 {

namespace {

namespace cg = cooperative_groups;

// Planner allowances, in sub-items of streaming: a shared-memory reduction
// per tile when warps share it, a workspace round trip per tile (fence and
// counter) and the last partial's extra round trips at the end of a launch;
// the cluster form's end (two cluster barriers, which wait for the slowest of
// the cluster's CTAs, and nch partial reads per tile) as a base plus a part
// per chunk (fitted to lone-call times of the 8B / 32B decode shapes at
// M = 2, 4, 8 over every chunk count in both forms).
#ifndef NVFP4_SPLITK_COST_GROUP
#define NVFP4_SPLITK_COST_GROUP 0.5
#endif
#ifndef NVFP4_SPLITK_COST_FLUSH
#define NVFP4_SPLITK_COST_FLUSH 3.0
#endif
#ifndef NVFP4_SPLITK_COST_TAIL
#define NVFP4_SPLITK_COST_TAIL 3.0
#endif
#ifndef NVFP4_SPLITK_COST_CLUSTER
#define NVFP4_SPLITK_COST_CLUSTER 1.0
#endif
#ifndef NVFP4_SPLITK_COST_CLUSTER_CHUNK
#define NVFP4_SPLITK_COST_CLUSTER_CHUNK 0.5
#endif
#ifndef NVFP4_SPLITK_STAGES
#define NVFP4_SPLITK_STAGES 3
#endif
constexpr int kWarps = 16;                    // warps per CTA (one CTA per SM)
constexpr int kStages = NVFP4_SPLITK_STAGES;  // sub-items per warp in its shared-memory ring
constexpr int kSub = 256;        // elements of K per sub-item
constexpr int kSlotBytes = 16 * 128 + 16 * 16;  // codes and scales of one 16-row sub-item
constexpr size_t kRingSmem = (size_t)kWarps * kStages * kSlotBytes;
constexpr size_t kFragSmem = 64 * 1024;  // activation fragments: 2 M bytes per K element
constexpr size_t kGroupSmem = 2 * kWarps * 32 * 16;  // partial tiles of the warp groups
constexpr size_t kMaxSmem = kRingSmem + kFragSmem + kGroupSmem;
constexpr int kMaxClusterChunks = 8;  // portable cluster size

// Longest chunk whose fragments (M rows, 2 bytes per element) fit.
__host__ __device__ constexpr int64_t max_chunk(int64_t m)
{
    return (int64_t)(kFragSmem / (2 * m)) / kSub * kSub;
}

struct SplitkParams {
    const uint8_t* xq;
    const uint8_t* xs;
    const float* xg;
    const uint8_t* wq;
    const uint8_t* ws;
    const float* wg;
    OutY y;
    float4* part;     // [tiles][nchunks][32 lanes] partial tiles (nchunks > 1)
    unsigned* count;  // [tiles] partials stored so far; zero between calls
    int m;
    int64_t n;
    int64_t k;
    int kc;     // longest chunk, elements (sizes the fragment area)
    int sub_q;  // sub-items of a short chunk
    int sub_r;  // chunks (the first ones) one sub-item longer
    int grp;    // warps that share a tile (1, 2, 4 or 8), splitting its chunk
    int maxj;  // cluster form: partial slots per warp group (its most tiles)
};

// One sub-item of a lane, read from its ring slot: 16 + 16 code bytes of rows
// g and g + 8 and their four block scales each (two scale bytes per register,
// as the E4M3-pair conversion takes them).
struct Sub {
    uint4 a0, a1;       // row g
    uint4 b0, b1;       // row g + 8
    uint32_t sa0, sa1;  // row g scale bytes {2t, 2t+1} and {8+2t, 9+2t}
    uint32_t sb0, sb1;  // row g + 8, same
};

// Code word w (0..7) of a lane with quad position t holds the 8 elements at
// offset (w < 4 ? 0 : 128) + 32 t + 8 (w & 3) of the sub-item: words 0..3 are
// its first 16 bytes, 4..7 the second; the activation fragments follow the
// same order.

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most kStages - 1 of this thread's copy groups are pending.
__device__ __forceinline__ void cp_async_wait_oldest()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(kStages - 1) : "memory");
}

template <bool PDL, bool CLUSTER>
__global__ void __launch_bounds__(kWarps * 32, 1) splitk_kernel(const SplitkParams prm)
{
    // [kWarps][kStages] sub-item slots of the warps' copy rings, then
    // [kc / 256][8 words][4 M lanes] activation fragments, then (grp > 1)
    // [2][kWarps][32 lanes] float4 partial tiles of the warp groups, then
    // (cluster form) [kWarps / grp][maxj][32 lanes] float4 chunk partials
    extern __shared__ __align__(16) unsigned char smem[];
    if constexpr (PDL)
        asm volatile("griddepcontrol.launch_dependents;");

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int chunk = blockIdx.x, nch = gridDim.x;
    const int64_t n = prm.n, kh = prm.k / 2, kb = prm.k / 16;
    const int nsub = prm.sub_q + (chunk < prm.sub_r ? 1 : 0);
    const int64_t k0 = ((int64_t)chunk * prm.sub_q + (chunk < prm.sub_r ? chunk : prm.sub_r)) * kSub;
    const int64_t ntiles = (n + 15) / 16;
    // warp group gi (grp warps) owns tiles; warp rank r of the group takes
    // sub-items r, r + grp, ... of each tile's chunk
    const int G = prm.grp, gi = warp / G, r = warp - gi * G, ngrp = kWarps / G;
    const int64_t tile0 = (int64_t)blockIdx.y * ngrp + gi;
    const int64_t tstride = (int64_t)gridDim.y * ngrp;
    // this warp's sub-items (fits an int: the planner takes N < 2^27)
    const int mytiles = tile0 < ntiles ? (int)((ntiles - 1 - tile0) / tstride) + 1 : 0;
    const int per_tile = nsub / G;  // sub-items of each warp per tile
    const int nitems = mytiles * per_tile;
    int copies_left = nitems;
    unsigned char* slots = smem + (size_t)warp * kStages * kSlotBytes;
    const uint32_t slots_s = (uint32_t)__cvta_generic_to_shared(slots);
    uint4* xfrag = reinterpret_cast<uint4*>(smem + kRingSmem);

    // copy cursor: the next sub-item's tile and index, and this lane's source
    // addresses in rows g and g + 8 of that tile.  Rows past n copy row n - 1
    // instead (they only reach D rows that are never stored); sub-items past
    // the warp's last tile copy nothing (an empty group keeps the count).
    int64_t f_tile = tile0;
    int f_sub = r;
    const uint8_t *fa, *fb, *qa, *qb;
    auto point = [&](int64_t tile) {
        const int64_t row = tile * 16 + g;
        const int64_t ra = row < n ? row : n - 1, rb = row + 8 < n ? row + 8 : n - 1;
        const int64_t c0 = k0 + (int64_t)r * kSub;
        fa = prm.wq + ra * kh + c0 / 2 + 16 * t;
        fb = prm.wq + rb * kh + c0 / 2 + 16 * t;
        qa = prm.ws + ra * kb + c0 / 16 + 4 * t;
        qb = prm.ws + rb * kb + c0 / 16 + 4 * t;
    };
    point(tile0);
    // Slot layout: four 512-byte planes of code bytes (rows g | g + 8, first
    // | second 16 bytes; lane l at 16 l, so every access is conflict-free),
    // then the 16 scale bytes of each of the 16 rows; lane (g, t) copies
    // scale bytes [4t, 4t + 4) of rows g and g + 8, the quad the whole row.
    auto issue = [&](int s) {
        if (copies_left > 0) {
            --copies_left;
            const uint32_t d = slots_s + (uint32_t)(s * kSlotBytes);
            cp_async16(d + 0 * 512 + lane * 16, fa);
            cp_async16(d + 1 * 512 + lane * 16, fa + 64);
            cp_async16(d + 2 * 512 + lane * 16, fb);
            cp_async16(d + 3 * 512 + lane * 16, fb + 64);
            cp_async4(d + 2048 + g * 16 + 4 * t, qa);
            cp_async4(d + 2048 + (8 + g) * 16 + 4 * t, qb);
            f_sub += G;
            if (f_sub >= nsub) {
                f_sub = r;
                f_tile += tstride;
                point(f_tile);
            } else {
                fa += G * (kSub / 2);
                fb += G * (kSub / 2);
                qa += G * (kSub / 16);
                qb += G * (kSub / 16);
            }
        }
        cp_async_commit();
    };
    auto read_slot = [&](int s) {
        const unsigned char* d = slots + s * kSlotBytes;
        Sub sl;
        sl.a0 = *reinterpret_cast<const uint4*>(d + 0 * 512 + lane * 16);
        sl.a1 = *reinterpret_cast<const uint4*>(d + 1 * 512 + lane * 16);
        sl.b0 = *reinterpret_cast<const uint4*>(d + 2 * 512 + lane * 16);
        sl.b1 = *reinterpret_cast<const uint4*>(d + 3 * 512 + lane * 16);
        sl.sa0 = *reinterpret_cast<const unsigned short*>(d + 2048 + g * 16 + 2 * t);
        sl.sa1 = *reinterpret_cast<const unsigned short*>(d + 2048 + g * 16 + 8 + 2 * t);
        sl.sb0 = *reinterpret_cast<const unsigned short*>(d + 2048 + (8 + g) * 16 + 2 * t);
        sl.sb1 = *reinterpret_cast<const unsigned short*>(d + 2048 + (8 + g) * 16 + 8 + 2 * t);
        return sl;
    };

#pragma unroll
    for (int s = 0; s < kStages; ++s)
        issue(s);

    // the activations are written by the previous kernel on the stream
    if constexpr (PDL)
        asm volatile("griddepcontrol.wait;" ::: "memory");
    const int M = prm.m;
    // Activation fragments of the chunk, for the M real columns only: lane
    // (g, t) with g < M holds word w of sub-item `sub` at
    // xfrag[(sub * 8 + w) * LW + lane], LW = 4 M lanes per word (the other
    // lanes' B fragments are not stored).  Unit hs = 2 sub + h of the chunk
    // is 128 elements of each of the M rows; warp hs % 8 decodes it, lane
    // (gg, tt) < LW taking the 32 elements (16 code bytes, two block scales)
    // that fill its words 4h .. 4h + 3.  A warp issues the loads of all its
    // units before it decodes any (one round trip to L2).
    const int LW = 4 * M;
    if (lane < LW) {
        constexpr int kUnroll = 4;
        const int nhs = nsub * 2, gg = lane >> 2, tt = lane & 3;
        const uint8_t* xq_row = prm.xq + gg * kh + (k0 + 32 * tt) / 2;
        const uint8_t* xs_row = prm.xs + gg * kb + (k0 + 32 * tt) / 16;
        for (int base = warp; base < nhs; base += kUnroll * kWarps) {
            uint4 c[kUnroll];
            uint32_t sc[kUnroll];
#pragma unroll
            for (int j = 0; j < kUnroll; ++j) {
                const int hs = base + j * kWarps;
                c[j] = make_uint4(0u, 0u, 0u, 0u);
                sc[j] = 0u;
                if (hs < nhs) {  // element offset hs * 128 within the chunk
                    c[j] = __ldg(reinterpret_cast<const uint4*>(xq_row + hs * 64));
                    sc[j] = __ldg(reinterpret_cast<const unsigned short*>(xs_row + hs * 8));
                }
            }
#pragma unroll
            for (int j = 0; j < kUnroll; ++j) {
                const int hs = base + j * kWarps;
                if (hs >= nhs)
                    break;
                const uint32_t s01 = e4m3x2_to_f16x2_bits(sc[j]);
                const uint32_t words[4] = {c[j].x, c[j].y, c[j].z, c[j].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t scl = q < 2 ? f16x2_dup_lo(s01) : f16x2_dup_hi(s01);
                    uint32_t hq[4];
                    e2m1x8_to_f16(words[q], hq);
                    // word 4 (hs & 1) + q of sub-item hs / 2
                    xfrag[(hs * 4 + q) * LW + lane] =
                        make_uint4(f16x2_mul(hq[0], scl), f16x2_mul(hq[1], scl),
                                   f16x2_mul(hq[2], scl), f16x2_mul(hq[3], scl));
                }
            }
        }
    }
    __syncthreads();
    const float gxw = __fmul_rn(__ldg(prm.xg), __ldg(prm.wg));

    // two accumulator sets (the first and second MMA of each word) halve the
    // dependent MMA chain; they are added at the end of the tile
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};

    // 16 MMAs over one sub-item: word w of the lane's codes (rows g, g + 8)
    // feeds MMAs 2w and 2w + 1 with the word's block scale folded in.  Lanes
    // of columns g >= M read another column's fragment: B column g only
    // reaches D column g, which is never stored.
    const int lane_b = lane % LW;
    auto consume = [&](const Sub& sl, const uint4* bsrc) {
        const uint32_t sa01 = e4m3x2_to_f16x2_bits(sl.sa0);
        const uint32_t sa23 = e4m3x2_to_f16x2_bits(sl.sa1);
        const uint32_t sb01 = e4m3x2_to_f16x2_bits(sl.sb0);
        const uint32_t sb23 = e4m3x2_to_f16x2_bits(sl.sb1);
        const uint32_t wa[8] = {sl.a0.x, sl.a0.y, sl.a0.z, sl.a0.w,
                                sl.a1.x, sl.a1.y, sl.a1.z, sl.a1.w};
        const uint32_t wb[8] = {sl.b0.x, sl.b0.y, sl.b0.z, sl.b0.w,
                                sl.b1.x, sl.b1.y, sl.b1.z, sl.b1.w};
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const uint32_t pa = w < 4 ? sa01 : sa23, pb = w < 4 ? sb01 : sb23;
            const uint32_t sA = (w & 2) ? f16x2_dup_hi(pa) : f16x2_dup_lo(pa);
            const uint32_t sB = (w & 2) ? f16x2_dup_hi(pb) : f16x2_dup_lo(pb);
            uint32_t ha[4], hb[4];
            e2m1x8_to_f16(wa[w], ha);
            e2m1x8_to_f16(wb[w], hb);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                ha[q] = f16x2_mul(ha[q], sA);
                hb[q] = f16x2_mul(hb[q], sB);
            }
            const uint4 xb = bsrc[w * LW];
            mma_m16n8k16(acc, ha[0], hb[0], ha[1], hb[1], xb.x, xb.y);
            mma_m16n8k16(acc2, ha[2], hb[2], ha[3], hb[3], xb.z, xb.w);
        }
    };

    // Y of a tile's 16 rows x M columns from this lane's four sums.
    auto store_tile = [&](int64_t tile, float v0, float v1, float v2, float v3) {
        const int64_t r0 = tile * 16 + g, r1 = r0 + 8;
        const int c0 = 2 * t, c1 = c0 + 1;
        if (c0 < M) {
            if (r0 < n)
                store_y(prm.y, c0 * n + r0, v0 * gxw);
            if (r1 < n)
                store_y(prm.y, c0 * n + r1, v2 * gxw);
        }
        if (c1 < M) {
            if (r0 < n)
                store_y(prm.y, c1 * n + r0, v1 * gxw);
            if (r1 < n)
                store_y(prm.y, c1 * n + r1, v3 * gxw);
        }
    };

    // cluster form: the chunk partial of the group's jt-th tile
    float4* pstore = reinterpret_cast<float4*>(
        smem + kRingSmem + (size_t)prm.kc * 2 * M + (G > 1 ? kGroupSmem : 0));

    // End of a tile's chunk (one warp per tile, the group's jt-th): Y
    // directly, or the cluster form's shared-memory slot, or the workspace
    // and, for the last partial of the tile, the fixed-order sum.
    auto flush = [&](int64_t tile, int jt, float v0, float v1, float v2, float v3) {
        if (CLUSTER && nch > 1) {
            pstore[(gi * prm.maxj + jt) * 32 + lane] = make_float4(v0, v1, v2, v3);
            return;
        }
        if (nch > 1) {
            float4* slot = prm.part + tile * nch * 32 + lane;
            __stcg(slot + chunk * 32, make_float4(v0, v1, v2, v3));
            __threadfence();
            __syncwarp();
            unsigned prev = 0u;
            if (lane == 0) {
                __threadfence();
                prev = atomicAdd(prm.count + tile, 1u);
            }
            prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
            if (prev != (unsigned)nch - 1)
                return;
            __threadfence();
            __syncwarp();
            // chunk order; the loads of 4 partials are issued before their sums
            float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int c0 = 0; c0 < nch; c0 += 4) {
                float4 p[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (c0 + j < nch)
                        p[j] = __ldcg(slot + (c0 + j) * 32);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (c0 + j < nch) {
                        s.x += p[j].x;
                        s.y += p[j].y;
                        s.z += p[j].z;
                        s.w += p[j].w;
                    }
            }
            v0 = s.x;
            v1 = s.y;
            v2 = s.z;
            v3 = s.w;
            if (lane == 0)
                atomicExch(prm.count + tile, 0u);
        }
        store_tile(tile, v0, v1, v2, v3);
    };

    // End of a warp's share of a tile: with warp groups, the group's warps
    // leave their partials in shared memory (double-buffered, so one barrier
    // per tile suffices) and rank 0 adds them in rank order and flushes.
    float4* red = reinterpret_cast<float4*>(xfrag + nsub * 8 * LW);  // after the fragments
    int rbuf = 0;
    auto tile_end = [&](int64_t tile, int jt) {
        float v0 = acc[0] + acc2[0], v1 = acc[1] + acc2[1], v2 = acc[2] + acc2[2],
              v3 = acc[3] + acc2[3];
        if (G > 1) {
            red[(rbuf * kWarps + warp) * 32 + lane] = make_float4(v0, v1, v2, v3);
            asm volatile("bar.sync %0, %1;" ::"r"(1 + gi), "r"(G * 32) : "memory");
            const float4* src = red + (rbuf * kWarps + gi * G) * 32 + lane;
            rbuf ^= 1;
            if (r != 0)
                return;
            float4 s4 = src[0];
            for (int q = 1; q < G; ++q) {
                const float4 p = src[q * 32];
                s4.x += p.x;
                s4.y += p.y;
                s4.z += p.z;
                s4.w += p.w;
            }
            v0 = s4.x;
            v1 = s4.y;
            v2 = s4.z;
            v3 = s4.w;
        }
        flush(tile, jt, v0, v1, v2, v3);
    };

    int64_t c_tile = tile0;
    const int b_first = r * 8 * LW, b_step = G * 8 * LW;  // fragment offsets of this warp's sub-items
    int c_b = b_first, c_left = per_tile, c_j = 0;
    const uint4* xb = xfrag + lane_b;
    for (int e = 0; e < nitems; e += kStages) {
#pragma unroll
        for (int s = 0; s < kStages; ++s) {
            if (e + s < nitems) {
                // the oldest group (this slot) is complete for this lane; the
                // warp barrier makes every lane's copies (the shared scale
                // rows) visible to the others
                cp_async_wait_oldest();
                __syncwarp();
                consume(read_slot(s), xb + c_b);
                __syncwarp();  // every lane is done reading the slot
                issue(s);
                c_b += b_step;
                if (--c_left == 0) {
                    tile_end(c_tile, c_j++);
                    acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
                    acc2[0] = acc2[1] = acc2[2] = acc2[3] = 0.f;
                    c_b = b_first;
                    c_left = per_tile;
                    c_tile += tstride;
                }
            }
        }
    }
    // no copy is left in flight: every group issued past the last sub-item
    // was empty

    if constexpr (CLUSTER) {
        if (nch > 1) {
            // Every partial of the cluster's tile set is in its CTA's shared
            // memory once all CTAs pass the barrier.  Slot e = (group, j) of
            // every rank holds that rank's chunk of the same tile; the
            // cluster's warps take the slots in turn and sum the nch partials
            // from zero in chunk order, as the workspace form does.
            cg::cluster_group cl = cg::this_cluster();
            cl.sync();
            const int nent = ngrp * prm.maxj;
            for (int e = chunk * kWarps + warp; e < nent; e += nch * kWarps) {
                const int egi = e / prm.maxj, ej = e - egi * prm.maxj;
                const int64_t tile = (int64_t)blockIdx.y * ngrp + egi + (int64_t)ej * tstride;
                if (tile >= ntiles)
                    continue;
                float4 p[kMaxClusterChunks];
#pragma unroll
                for (int c = 0; c < kMaxClusterChunks; ++c)
                    if (c < nch)
                        p[c] = *cl.map_shared_rank(pstore + e * 32 + lane, (unsigned)c);
                float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int c = 0; c < kMaxClusterChunks; ++c)
                    if (c < nch) {
                        s4.x += p[c].x;
                        s4.y += p[c].y;
                        s4.z += p[c].z;
                        s4.w += p[c].w;
                    }
                store_tile(tile, s4.x, s4.y, s4.z, s4.w);
            }
            cl.sync();  // no CTA leaves while another may still read its partials
        }
    }
}

struct SplitkPlan {
    int kc, nch, grp;  // longest chunk (elements), chunks, warps per tile
    int64_t cy;
    bool cluster;  // partials summed through distributed shared memory
    int maxj;      // cluster form: partial slots per warp group
};

// Workspace layout: the per-tile counters in the first counter_region(size)
// bytes, the partial tiles after them.  The split depends only on the
// workspace's size, never on the shape, so calls of different shapes that
// share one workspace keep each other's partials out of the counters (which
// must stay zero between calls).  A split call has at least two 512-byte
// partials per tile, so its counters (4 bytes per tile) always fit.
int64_t counter_region(int64_t ws_bytes)
{
    return (ws_bytes / 128 + 255) / 256 * 256;
}

bool plan_fits(int64_t ntiles, int nch, int64_t ws_bytes)
{
    if (nch <= 1)
        return true;
    const int64_t p0 = counter_region(ws_bytes);
    const int64_t parts = ntiles * nch * 32 * (int64_t)sizeof(float4);
    return ntiles * 4 <= p0 && parts <= ws_bytes - p0;
}

int64_t workspace_bytes_for(int64_t ntiles, int nch)
{
    if (nch <= 1)
        return 0;
    const int64_t parts = ntiles * nch * 32 * (int64_t)sizeof(float4);
    int64_t ws = (parts + parts / 127 + 511) / 256 * 256;
    while (!plan_fits(ntiles, nch, ws))
        ws += 256;
    return ws;
}

// CTAs of the kernel resident on the current device (the occupancy at the
// largest chunk; the shared memory limit is raised first, since the query
// counts against the limit in force).
int64_t resident_ctas()
{
    const int dev = current_device();
    const size_t smem = kMaxSmem;
    int per_sm = 0;
    if (ensure_smem_limit(splitk_kernel<false, false>, smem, dev) != cudaSuccess ||
        ensure_smem_limit(splitk_kernel<true, false>, smem, dev) != cudaSuccess ||
        cached_occupancy(splitk_kernel<true, false>, kWarps * 32, smem, 0, dev, &per_sm) !=
            cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    return (int64_t)device_sm_count(dev) * per_sm;
}

// Largest dynamic shared memory a CTA may opt into on the current device.
size_t smem_optin()
{
    const int dev = current_device();
    static std::mutex mu;
    static std::unordered_map<int, size_t> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it != cache.end())
        return it->second;
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        v = 0;
    cache[dev] = (size_t)v;
    return (size_t)v;
}

// Clusters of `nch` CTAs of the cluster form that run at once on the current
// device (0 if the query fails).  Every CTA needs more than half an SM's
// shared memory, so one per SM whatever its exact size: the query is made at
// the opt-in maximum.
int64_t resident_clusters(int nch)
{
    const int dev = current_device();
    const size_t smem = smem_optin();
    int v = 0;
    if (smem < kMaxSmem ||
        ensure_smem_limit(splitk_kernel<false, true>, smem, dev) != cudaSuccess ||
        ensure_smem_limit(splitk_kernel<true, true>, smem, dev) != cudaSuccess ||
        cached_occupancy(splitk_kernel<true, true>, kWarps * 32, smem, nch, dev, &v) !=
            cudaSuccess)
        return 0;
    return v;
}

size_t plan_smem(const SplitkPlan& p, int64_t m)
{
    return kRingSmem + (size_t)p.kc * 2 * m + (p.grp > 1 ? kGroupSmem : 0) +
           (p.cluster ? (size_t)(kWarps / p.grp) * p.maxj * 32 * sizeof(float4) : 0);
}

// Candidates: nch chunks (the longest at most max_chunk(m)); warps per tile
// grp 1, 2, 4, 8 or 16 dividing every chunk's sub-items (so grp = 1 when the
// chunks are unequal); each split candidate in its workspace form (when its
// partials fit `ws_limit`) and in its cluster form (nch <= 8, the partials
// within the shared memory).  The cost of a candidate, in units of one
// sub-item of streaming, is the busiest warp's sub-items plus allowances for
// what adds latency: a shared-memory reduction per tile when warps share it;
// in the workspace form one round trip per tile and the last partial's at the
// end; in the cluster form its end-of-launch reduction.  The cheapest wins;
// ties go to the earlier candidate (fewer chunks, fewer warps per tile, the
// workspace form).
bool search_splitk(int64_t m, int64_t n, int64_t k, int64_t ws_limit, SplitkPlan* out)
{
    if (m < 1 || m > 8 || n < 1 || n >= (int64_t(1) << 27) || k < kSub || k % kSub != 0)
        return false;
    const int64_t slots = resident_ctas();
    const int64_t ntiles = (n + 15) / 16;
    const int64_t subs = k / kSub, len_max = max_chunk(m) / kSub;
    bool found = false;
    double best = 0.0;
    for (int64_t nch = (subs + len_max - 1) / len_max; nch <= subs && nch <= 65535; ++nch) {
        const int64_t q = subs / nch, r = subs % nch, len = q + (r ? 1 : 0);
        for (int form = 0; form < 2; ++form) {
            const bool cluster = form == 1;
            if (nch == 1 && cluster)
                continue;
            if (!cluster && !plan_fits(ntiles, (int)nch, ws_limit))
                continue;
            if (cluster && nch > kMaxClusterChunks)
                continue;
            const int64_t clusters = cluster ? resident_clusters((int)nch) : 0;
            if (cluster && clusters < 1)
                continue;
            for (int grp = 1; grp <= kWarps; grp *= 2) {
                if (q % grp || (r && grp > 1))
                    continue;
                const int64_t ngrp = kWarps / grp;
                int64_t cy = cluster ? clusters : slots / nch;
                const int64_t cy_max = (ntiles + ngrp - 1) / ngrp;
                if (cy > cy_max)
                    cy = cy_max;
                if (cy < 1)
                    cy = 1;
                const int64_t per_group = (ntiles + cy * ngrp - 1) / (cy * ngrp);
                const SplitkPlan cand = {(int)(len * kSub), (int)nch, grp, cy, cluster,
                                         (int)per_group};
                if (cluster && plan_smem(cand, m) > smem_optin())
                    continue;
                const double per_tile = (double)(len / grp) +
                                        (grp > 1 ? NVFP4_SPLITK_COST_GROUP : 0.0) +
                                        (nch > 1 && !cluster ? NVFP4_SPLITK_COST_FLUSH : 0.0);
                const double tail =
                    nch <= 1  ? 0.0
                    : cluster ? NVFP4_SPLITK_COST_CLUSTER + NVFP4_SPLITK_COST_CLUSTER_CHUNK * nch
                              : NVFP4_SPLITK_COST_TAIL;
                const double cost = (double)per_group * per_tile + tail;
                if (!found || cost < best) {
                    found = true;
                    best = cost;
                    *out = cand;
                }
            }
        }
    }
    return found;
}

// The plan of a call offering `ws_limit` bytes of workspace: the best of the
// candidates it can run (with any workspace at least the size that
// splitk_workspace_bytes reports, the best of all).  Cached per device,
// shape and offer, so that a launch plans once.
struct PlanKey {
    int dev;
    int64_t m, n, k, ws;
    bool operator==(const PlanKey& o) const
    {
        return dev == o.dev && m == o.m && n == o.n && k == o.k && ws == o.ws;
    }
};
struct PlanKeyHash {
    size_t operator()(const PlanKey& p) const
    {
        size_t h = (size_t)p.dev;
        h = h * 1000003u ^ (size_t)p.m;
        h = h * 1000003u ^ (size_t)p.n;
        h = h * 1000003u ^ (size_t)p.k;
        h = h * 1000003u ^ (size_t)p.ws;
        return h;
    }
};

bool plan_splitk(int64_t m, int64_t n, int64_t k, int64_t ws_limit, SplitkPlan* out)
{
    static std::mutex mu;
    static std::unordered_map<PlanKey, std::pair<bool, SplitkPlan>, PlanKeyHash> cache;
    const PlanKey key{current_device(), m, n, k, ws_limit};
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            *out = it->second.second;
            return it->second.first;
        }
    }
    SplitkPlan p = {};
    const bool ok = search_splitk(m, n, k, ws_limit, &p);
    std::lock_guard<std::mutex> lock(mu);
    if (cache.size() > 4096)
        cache.clear();
    cache[key] = {ok, p};
    *out = p;
    return ok;
}

template <bool PDL, bool CLUSTER>
cudaError_t launch_t(const GemmArgs& a, const SplitkPlan& p, void* workspace, int64_t ws_bytes)
{
    const size_t smem = plan_smem(p, a.m);
    auto kern = splitk_kernel<PDL, CLUSTER>;
    const int dev = current_device();
    if (smem > 48 * 1024) {
        const cudaError_t e = ensure_smem_limit(kern, CLUSTER ? smem_optin() : kMaxSmem, dev);
        if (e != cudaSuccess)
            return e;
    }
    const int subs = (int)(a.k / kSub);
    SplitkParams prm = {a.xq, a.xs, a.xg, a.wq, a.ws, a.wg, a.y, nullptr,
                        nullptr, a.m, a.n, a.k, p.kc, subs / p.nch, subs % p.nch,
                        p.grp, p.maxj};
    if (p.nch > 1 && !CLUSTER) {
        unsigned char* base = static_cast<unsigned char*>(workspace);
        prm.count = reinterpret_cast<unsigned*>(base);
        prm.part = reinterpret_cast<float4*>(base + counter_region(ws_bytes));
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.nch, (unsigned)p.cy, 1);
    cfg.blockDim = dim3(kWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (CLUSTER) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)p.nch;
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

// Scratch of the allocation-free entry point: a fixed array in the module's
// device image, zero when the module is loaded.  Every call on a device
// shares it, so calls that may overlap in time race.
constexpr int64_t kStaticScratchBytes = int64_t(4) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of the static scratch on the current device, looked up
// once per device.  Its counter region needs no clearing: the array is zero
// when the module loads and every completed call leaves the counters zero
// (a memset here would also race with a call still running on another
// stream).  A launch that fails drops the cached address, so that it is
// looked up again on the next call (after a context reset, for instance).
std::mutex g_scratch_mu;
std::unordered_map<int, void*> g_scratch_addr;

cudaError_t static_scratch(void** out)
{
    const int dev = current_device();
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    auto it = g_scratch_addr.find(dev);
    if (it != g_scratch_addr.end()) {
        *out = it->second;
        return cudaSuccess;
    }
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess)
        return e;
    g_scratch_addr[dev] = p;
    *out = p;
    return cudaSuccess;
}

void forget_static_scratch()
{
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    g_scratch_addr.erase(current_device());
}

}  // namespace

int64_t splitk_static_scratch_bytes()
{
    return kStaticScratchBytes;
}

bool splitk_static_fits(int64_t m, int64_t n, int64_t k)
{
    SplitkPlan p;
    return plan_splitk(m, n, k, INT64_MAX, &p) &&
           (p.cluster || plan_fits((n + 15) / 16, p.nch, kStaticScratchBytes));
}

cudaError_t launch_gemm_splitk_static(const GemmArgs& a, bool pdl)
{
    void* scratch = nullptr;
    const cudaError_t e = static_scratch(&scratch);
    if (e != cudaSuccess)
        return e;
    const cudaError_t l = launch_gemm_splitk(a, pdl, scratch, kStaticScratchBytes);
    if (l != cudaSuccess)
        forget_static_scratch();
    return l;
}

bool splitk_shape_ok(int64_t m, int64_t k)
{
    return m >= 1 && m <= 8 && k >= kSub && k % kSub == 0;
}

bool splitk_plan_ok(int64_t m, int64_t n, int64_t k, int64_t workspace_bytes)
{
    SplitkPlan p;
    return plan_splitk(m, n, k, workspace_bytes, &p);
}

int64_t splitk_workspace_bytes(int64_t m, int64_t n, int64_t k)
{
    SplitkPlan p;
    if (!plan_splitk(m, n, k, INT64_MAX, &p) || p.cluster)
        return 0;
    return workspace_bytes_for((n + 15) / 16, p.nch);
}

cudaError_t launch_gemm_splitk(const GemmArgs& a, bool pdl, void* workspace,
                               int64_t workspace_bytes)
{
    SplitkPlan p;
    if (!plan_splitk(a.m, a.n, a.k, workspace ? workspace_bytes : 0, &p))
        return cudaErrorInvalidValue;
    if (p.cluster)
        return pdl ? launch_t<true, true>(a, p, nullptr, 0) : launch_t<false, true>(a, p, nullptr, 0);
    return pdl ? launch_t<true, false>(a, p, workspace, workspace_bytes)
               : launch_t<false, false>(a, p, workspace, workspace_bytes);
}

}  // namespace nvfp4
