// gemm_tc.cu -- small-M W4A4 linears on the fifth-generation tensor cores:
// tcgen05.mma kind::mxf4nvf4 (E2M1 x E2M1 with one UE4M3 scale per 16
// elements of K on each side, FP32 accumulation in tensor memory), for M up
// to 32.  The ReSET README ("Core components" item 2) leaves the tensor cores
// aside at M <= 8 because a 128-row MMA tile would be at most 8/128 occupied;
// here the operands are swapped -- 128 WEIGHT rows fill the MMA's M side and
// the M activation rows are its N side (16 or 32, rows past M unused) -- so
// the tile is full and the MMA consumes FP4 weights and their scales directly:
// no decode, no scale fold and no FMA per weight element on the CUDA cores.
//
// One persistent CTA per SM streams a contiguous range of the 128-row weight
// tiles of a list of independent linears (one linear is a list of one), K
// whole per tile, through an 8-stage shared-memory ring.  Warp roles:
//   warp 0      one thread issues each stage's 128 x 256 weight-code copy: one
//               contiguous 16 KB cp.async.bulk with tile-major weights (laid
//               out in the swizzled shared-memory image when packed), a TMA
//               box (cp.async.bulk.tensor, 128-byte swizzle) with row-major ones;
//   warp 1      allocates tensor memory; one thread issues the MMAs: four
//               K = 64 MMAs per stage into the tile's accumulator (two
//               accumulators alternate, so the epilogue of one tile overlaps
//               the next), tcgen05.commit frees the stage and, after the last
//               stage, hands the accumulator to the epilogue;
//   warps 2..5  per stage: the weight rows' and activation rows' block scales
//               into tensor memory (tcgen05.st) and the activation codes into
//               the stage's shared-memory slot (same swizzled layout as TMA
//               writes), loaded from global memory kPrefetch stages ahead;
//   warps 6..9  epilogue: the accumulator out of tensor memory (tcgen05.ld),
//               Y[m][row] = acc * gX * gW (FP32 or BF16).
//   warps 10..14 (N = 16 with tile-major weights) the stream warps: the last
//               tiles of every linear at M <= 8 on the legacy mma.sync path,
//               beside the tcgen05 stream (see below).
// Every wait is on an mbarrier with a clock budget: running out records
// NVFP4_DEVICE_WAIT_TIMEOUT in the library's status word, every role stops,
// the copies and MMAs already issued are drained (again bounded) and tensor
// memory is freed before the CTA exits.
//
// Layouts, measured on GB300 with in-bounds probes before this kernel was
// written: operand descriptors for K-major 128-byte-swizzled tiles (8-row
// atoms of 1024 bytes, the start address advanced by 32 bytes per K = 64
// step inside the atom); scale factors of A row r at tensor-memory lane r,
// column sfa + r / 32; those of B column n at lane 32 q + n of column sfb for
// every lane quarter q; byte j of a 32-bit cell is the j-th 16-element block
// of the MMA's K = 64.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "../../include/nvfp4.h"
#include "kernels.cuh"
#include "launch_cache.cuh"
#include "formats.cuh"
#include "mma_frag.cuh"

namespace nvfp4 {

namespace {

#ifndef NVFP4_TC_STAGES
#define NVFP4_TC_STAGES 8
#endif
constexpr int kStages = NVFP4_TC_STAGES;   // shared-memory ring
constexpr int kRows = 128;                 // weight rows per tile (the MMA's M)
constexpr int kStageK = 256;               // K elements per stage (128 code bytes a row)
constexpr int kABytes = kRows * 128;       // weight codes of a stage
// activation codes of a stage: N rows of 128 bytes (two or four 1024-byte swizzle atoms)
template <int NMMA>
__host__ __device__ constexpr int b_bytes()
{
    return NMMA * 128;
}
// Stages ahead of the copy being issued whose weights the producer asks L2
// to fetch (0: none), to keep DRAM reads in flight beyond what the
// shared-memory ring holds.  Measured on the 8B decode step it only adds
// contention (M = 1: 0.665 ms without, 0.674 / 0.685 / 1.05 ms at 8 / 16 /
// 32 stages ahead), so it is off.
#ifndef NVFP4_TC_L2_AHEAD
#define NVFP4_TC_L2_AHEAD 0
#endif
constexpr int kL2Ahead = NVFP4_TC_L2_AHEAD;

// Stages the scale / activation warps load ahead (measured on the decode
// step: 6 against 4, 0.691 against 0.703-0.746 ms at M = 8).
#ifndef NVFP4_TC_PREFETCH
#define NVFP4_TC_PREFETCH 6
#endif
constexpr int kPrefetch = NVFP4_TC_PREFETCH;
constexpr int kThreads = 320;              // 10 warps of the tensor-core roles
// Stream warps (N = 16 kernel, tile-major weights): warps beside the
// tensor-core roles that take the last tiles of every linear (a share of them,
// in per mille of each linear's tiles, per M) when M <= 8, so that the SM adds
// a second weight stream to the tcgen05 one.  kStreamWarps compute warps (32
// rows of a tile each) and one copy warp.
#ifndef NVFP4_TC_STREAM_WARPS
#define NVFP4_TC_STREAM_WARPS 4
#endif
// share of every linear's tiles (per mille, rounded) the stream warps take, per M
// (measured optima on the 8B decode step, set a little below where the
// stream warps would become the slower part)
#ifndef NVFP4_TC_STREAM_SHARE_1
#define NVFP4_TC_STREAM_SHARE_1 320
#endif
#ifndef NVFP4_TC_STREAM_SHARE_2
#define NVFP4_TC_STREAM_SHARE_2 270
#endif
#ifndef NVFP4_TC_STREAM_SHARE_3
#define NVFP4_TC_STREAM_SHARE_3 250
#endif
#ifndef NVFP4_TC_STREAM_SHARE_4
#define NVFP4_TC_STREAM_SHARE_4 245
#endif
#ifndef NVFP4_TC_STREAM_SHARE_5
#define NVFP4_TC_STREAM_SHARE_5 220
#endif
#ifndef NVFP4_TC_STREAM_SHARE_6
#define NVFP4_TC_STREAM_SHARE_6 225
#endif
#ifndef NVFP4_TC_STREAM_SHARE_7
#define NVFP4_TC_STREAM_SHARE_7 212
#endif
#ifndef NVFP4_TC_STREAM_SHARE_8
#define NVFP4_TC_STREAM_SHARE_8 200
#endif
constexpr int kStreamShare[9] = {0, NVFP4_TC_STREAM_SHARE_1, NVFP4_TC_STREAM_SHARE_2,
                                 NVFP4_TC_STREAM_SHARE_3, NVFP4_TC_STREAM_SHARE_4,
                                 NVFP4_TC_STREAM_SHARE_5, NVFP4_TC_STREAM_SHARE_6,
                                 NVFP4_TC_STREAM_SHARE_7, NVFP4_TC_STREAM_SHARE_8};
constexpr int kStreamWarps = NVFP4_TC_STREAM_WARPS;
static_assert(kStreamWarps * 32 == kRows, "a stream warp per 32 rows of a tile");
template <int NMMA, bool TILED>
__host__ __device__ constexpr bool has_stream()
{
    return NMMA == 16 && TILED;
}
template <int NMMA, bool TILED>
__host__ __device__ constexpr int tc_threads()
{
    return has_stream<NMMA, TILED>() ? kThreads + 32 * (kStreamWarps + 1) : kThreads;
}
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColSfa = 64;                       // 16 columns per ring slot
constexpr uint32_t kColSfb = kColSfa + 16 * kStages;   // 16 columns per ring slot
static_assert(kColSfb + 16 * kStages <= kTmemCols, "scale slots fit the tensor memory");
constexpr long long kWaitBudget = 2000000000LL;  // clock cycles a wait may take
constexpr int kSBytes = kRows * 16;        // weight block scales of a stage (tile-major layout)
constexpr int kCcSlots = 3;                  // the stream warps' ring
// a slot: a stage's codes, its scales, then the B fragments of the stage's 16
// m16n8k16 MMAs per 16 rows (8 words x 32 lanes of 16 bytes, the activations'
// block scales folded in), which the copy warp prepares
constexpr int kCcXOff = kABytes + kSBytes;
constexpr int kCcFragBytes = 8 * 32 * 16;
constexpr int kCcBytes = kCcXOff + kCcFragBytes;
// ring: weight codes and activation codes (the weight scales go through
// registers), then the stream warps' slots
template <int NMMA, bool TILED>
constexpr size_t smem_bytes()
{
    return (size_t)kStages * (kABytes + b_bytes<NMMA>()) +
           (has_stream<NMMA, TILED>() ? (size_t)kCcSlots * kCcBytes : 0) + 1024;  // + alignment
}

struct TcItem {
    const uint8_t* xq;
    const uint8_t* xs;
    const float* xg;
    const uint8_t* wq;  // tile-major weight codes (the row-major ones go through wmap)
    const uint8_t* ws;  // weight block scales: row-major, or tile-major
    const float* wg;
    void* y;
    int32_t n, k;
    int32_t s0;  // first stage of this linear in the launch's stage list
    int32_t ttiles;  // leading tiles on the tensor cores (the rows past them: stream warps)
};
static_assert(sizeof(TcItem) == 72, "TcItem layout");

struct TcParams {
    CUtensorMap wmap[kTcMaxItems];  // weight codes [n][k/2]: boxes of 128 bytes x 128 rows,
                                    // 128-byte swizzle
    TcItem item[kTcMaxItems];
    int32_t start[kTcMaxCtas + 1];  // first stage of each CTA; start[grid] = all stages
    unsigned* status;               // the library's device status word
    float* part;      // [2 grid][32][128] partial tiles of tiles split between CTAs (or null)
    unsigned* count;  // [grid] arrival counters of split tiles (zero between calls)
    int32_t count_items;
    int32_t m;
    int32_t y_bf16;
    int32_t grid;
};
static_assert(sizeof(TcParams) <= 32764, "kernel parameters are limited to 32764 bytes");

// ---- small PTX wrappers --------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile("{\n\t.reg .pred q;\n\tmbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(done)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return done != 0;
}

// Wait for phase `parity` of `bar` to complete, within the clock budget and
// while no other role has given up; false when it did not.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned* status)
{
    const long long t0 = clock64();
    while (!mbar_test(bar, parity)) {
        if (*abort_flag)
            return false;
        if (clock64() - t0 > kWaitBudget) {
            *abort_flag = 1;
            atomicOr(status, (unsigned)NVFP4_DEVICE_WAIT_TIMEOUT);
            return false;
        }
    }
    return true;
}

// K-major operand tile with 128-byte swizzle: 8-row atoms of 1024 bytes.
__device__ __forceinline__ uint64_t operand_desc(uint32_t saddr)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)1 << 16;            // leading byte offset (not used by this layout)
    d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset: one 8-row atom
    d |= (uint64_t)1 << 46;            // descriptor version
    d |= (uint64_t)2 << 61;            // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::mxf4nvf4: E2M1 A and B, K-major both,
// UE4M3 scales, M = 128, N = nmma.
__host__ __device__ constexpr uint32_t instr_desc(int nmma)
{
    return (1u << 7) | (1u << 10) | ((uint32_t)(nmma >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24);
}

// 16 bytes of a weight row's block scales (one stage); the next stage's 16
// share its 32-byte sector.  NVFP4_TC_SCALE_L2 asks L2 to fetch the
// surrounding 64, 128 or 256 bytes with the same access (0: no hint).
// Measured on the 8B decode step (GEMM launch, two runs each): no hint
// 662 / 695 us at M = 1 / 8, 64 bytes 661 / 662 us, 128 bytes no change,
// 256 bytes slower at M = 8; 64 it is.
#ifndef NVFP4_TC_SCALE_L2
#define NVFP4_TC_SCALE_L2 64
#endif
__device__ __forceinline__ uint4 ld_nc_u4(const void* p)
{
    uint4 v;
#if NVFP4_TC_SCALE_L2 == 64
    asm volatile("ld.global.nc.L1::no_allocate.L2::64B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
#elif NVFP4_TC_SCALE_L2 == 128
    asm volatile("ld.global.nc.L1::no_allocate.L2::128B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
#elif NVFP4_TC_SCALE_L2 == 256
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
#else
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
#endif
    return v;
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

// Position in a CTA's sequence of (linear, tile, stage).
struct Cursor {
    int item;
    int32_t tile;   // tile index within the linear
    int32_t st;     // stage within the tile
    int32_t nst;    // stages per tile of this linear (k / 256)
    int32_t tiles;  // tiles of this linear
};

__device__ __forceinline__ int item_of_stage(const TcParams& p, int32_t g)
{
    int i = 0, b = p.count_items - 1;
    while (i < b) {
        const int mid = (i + b + 1) >> 1;
        if (p.item[mid].s0 <= g)
            i = mid;
        else
            b = mid - 1;
    }
    return i;
}

__device__ __forceinline__ void cursor_at(Cursor& c, const TcParams& p, int32_t g)
{
    c.item = item_of_stage(p, g);
    const TcItem& it = p.item[c.item];
    c.nst = it.k / kStageK;
    c.tiles = it.ttiles;
    const int32_t local = g - it.s0;
    c.tile = local / c.nst;
    c.st = local - c.tile * c.nst;
}

__device__ __forceinline__ void cursor_next_tile(Cursor& c, const TcParams& p)
{
    c.st = 0;
    if (++c.tile >= c.tiles && c.item + 1 < p.count_items) {
        ++c.item;
        c.tile = 0;
        c.nst = p.item[c.item].k / kStageK;
        c.tiles = p.item[c.item].ttiles;
    }
}

__device__ __forceinline__ void cursor_next_stage(Cursor& c, const TcParams& p)
{
    if (++c.st >= c.nst)
        cursor_next_tile(c, p);
}

// The CTA whose stage range holds stage g.
__device__ __forceinline__ int cta_of_stage(const TcParams& p, int32_t g)
{
    int c = 0, b = p.grid - 1;
    while (c < b) {
        const int mid = (c + b + 1) >> 1;
        if (p.start[mid] <= g)
            c = mid;
        else
            b = mid - 1;
    }
    return c;
}

// What a scale / activation thread loads for one stage.
struct AuxLoad {
    uint4 sa;  // block scales of this thread's weight row (4 MMA K-steps)
    uint4 sb;  // block scales of activation row `lane` (lanes < M)
    uint4 b0;  // activation codes, chunk u
    uint4 b1;  // activation codes, chunk u + 128 (M > 16)
};

template <int NMMA, bool TILED>
__device__ __forceinline__ void aux_load(AuxLoad& a, const TcParams& p, const Cursor& c, int r,
                                         int lane, int u)
{
    const TcItem& it = p.item[c.item];
    const int32_t kb = it.k / 16, kh = it.k / 2;
    const int64_t row = (int64_t)c.tile * kRows + r;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    if constexpr (TILED)  // the stage's 2 KB block, row r at 16 r (rows past n are zero)
        a.sa = ld_nc_u4(it.ws + ((size_t)c.tile * c.nst + c.st) * kSBytes + r * 16);
    else
        a.sa = row < it.n ? ld_nc_u4(it.ws + row * kb + c.st * 16) : z;
    a.sb = lane < p.m ? __ldg(reinterpret_cast<const uint4*>(it.xs + lane * kb + c.st * 16)) : z;
    a.b0 = u < p.m * 8
               ? __ldg(reinterpret_cast<const uint4*>(it.xq + (u >> 3) * kh + c.st * 128 +
                                                      (u & 7) * 16))
               : z;
    if constexpr (NMMA > 16)
        a.b1 = u + 128 < p.m * 8
                   ? __ldg(reinterpret_cast<const uint4*>(it.xq + ((u + 128) >> 3) * kh +
                                                          c.st * 128 + ((u + 128) & 7) * 16))
                   : z;
}

// ---- stream warps: whole tiles beside the tensor pipe -----------------------------
// The last tiles of every linear (tile-major weights, M <= 8) go to the stream
// warps: CTA b takes whole tiles, a contiguous range of them cut near an equal
// share of their stages.  The copy warp brings each stage's 16 KB of codes and
// 2 KB of scales (two contiguous blocks) into a ring of kCcSlots shared-memory
// slots and writes the stage's activation B fragments into the slot; compute
// warp w owns rows 32 w .. 32 w + 31 of the tile and runs the single-linear
// split-K kernel's MAC on them (E2M1 codes decoded to f16 with the 16-block
// scale folded in exactly, mma.sync m16n8k16, FP32 accumulation) -- the legacy
// MMA path, which the tcgen05 MMAs of the other warps leave free.  A tile's
// sums stay in the warp in stage order and go to Y at the tile's end: no
// partial leaves the CTA.
// The stream warps' stage list: the linears in order, tiles ttiles .. of each,
// K / 256 stages a tile.  The first tile boundary at or after stage `target`
// of that list (its length when `target` is past the end), so that CTA ranges
// cut there hold whole tiles.
__device__ int64_t cc_boundary(const TcParams& p, int64_t target)
{
    int64_t s = 0;
    for (int i = 0; i < p.count_items; ++i) {
        const TcItem& it = p.item[i];
        const int32_t nst = it.k / kStageK;
        const int64_t len = ((int64_t)(it.n + kRows - 1) / kRows - it.ttiles) * nst;
        if (target <= s)
            return s;
        if (target < s + len)
            return s + (target - s + nst - 1) / nst * nst;
        s += len;
    }
    return s;
}

struct CcCursor {
    int item;
    int32_t tile, st, nst, tiles;  // tile index within the linear; tiles of the linear
};

__device__ void cc_cursor_at(CcCursor& c, const TcParams& p, int64_t g)
{
    int64_t s = 0;
    for (int i = 0; i < p.count_items; ++i) {
        const TcItem& it = p.item[i];
        const int32_t nst = it.k / kStageK, tiles = (it.n + kRows - 1) / kRows;
        const int64_t len = (int64_t)(tiles - it.ttiles) * nst;
        if (g < s + len) {
            c.item = i;
            c.nst = nst;
            c.tiles = tiles;
            c.tile = it.ttiles + (int32_t)((g - s) / nst);
            c.st = (int32_t)((g - s) % nst);
            return;
        }
        s += len;
    }
    c.item = p.count_items;  // past the end
}

__device__ __forceinline__ void cc_next(CcCursor& c, const TcParams& p)
{
    if (++c.st < c.nst)
        return;
    c.st = 0;
    if (++c.tile < c.tiles)
        return;
    // the next linear that has stream tiles
    for (++c.item; c.item < p.count_items; ++c.item) {
        const TcItem& it = p.item[c.item];
        c.nst = it.k / kStageK;
        c.tiles = (it.n + kRows - 1) / kRows;
        c.tile = it.ttiles;
        if (c.tile < c.tiles)
            return;
    }
}

// The copy warp: stage i of the CTA's stream range into slot i % kCcSlots,
// once the compute warps have freed it (one lane issues the two bulk copies,
// every lane writes its B fragments of the stage into the slot and lane 0
// arrives a second time when they are there); then every copy in flight lands.
__device__ void cc_produce(const TcParams& p, int64_t lo, int64_t cnt, uint32_t sC0, uint8_t* sC,
                           uint64_t* full, uint64_t* empty, volatile int* abort_flag, int lane)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");  // x_q / x_s come from the producer
    CcCursor c;
    cc_cursor_at(c, p, lo);
    int64_t issued = 0;
    for (int64_t i = 0; i < cnt; ++i) {
        const int slot = (int)(i % kCcSlots);
        if (i >= kCcSlots &&
            !__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&empty[slot]),
                                               (uint32_t)(((i / kCcSlots) - 1) & 1), abort_flag,
                                               p.status)))
            break;
        const TcItem& it = p.item[c.item];
        const uint32_t fb = smem_u32(&full[slot]), dst = sC0 + (uint32_t)(slot * kCcBytes);
        if (lane == 0) {
            const size_t blk = (size_t)c.tile * c.nst + c.st;
            mbar_expect_tx(fb, kABytes + kSBytes);
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                ::"r"(dst), "l"(it.wq + blk * kABytes), "r"(kABytes), "r"(fb)
                : "memory");
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                ::"r"(dst + kABytes), "l"(it.ws + blk * kSBytes), "r"(kSBytes), "r"(fb)
                : "memory");
        }
        {
            // B fragments of the stage for the mma.sync MAC: lane (g, t) of
            // the compute warps takes, for code word w, the 8 elements at
            // (w < 4 ? 0 : 128) + 32 t + 8 (w & 3) of the stage from its rows;
            // its B fragment is activation row g at the same 8 elements, each
            // times its block scale (exact in f16), and zero for rows g >= M
            const int g = lane >> 2, t = lane & 3;
            uint4* fo = reinterpret_cast<uint4*>(sC + slot * kCcBytes + kCcXOff);
            if (g < p.m) {
                const uint8_t* xr = it.xq + g * (int64_t)(it.k / 2) + (int64_t)c.st * 128;
                const uint8_t* sr = it.xs + g * (int64_t)(it.k / 16) + (int64_t)c.st * 16;
                const uint4 v0 = __ldg(reinterpret_cast<const uint4*>(xr + 16 * t));
                const uint4 v1 = __ldg(reinterpret_cast<const uint4*>(xr + 64 + 16 * t));
                const uint32_t s01 = e4m3x2_to_f16x2_bits(
                    __ldg(reinterpret_cast<const unsigned short*>(sr + 2 * t)));
                const uint32_t s23 = e4m3x2_to_f16x2_bits(
                    __ldg(reinterpret_cast<const unsigned short*>(sr + 8 + 2 * t)));
                const uint32_t words[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    const uint32_t ps = w < 4 ? s01 : s23;
                    const uint32_t sc = (w & 2) ? f16x2_dup_hi(ps) : f16x2_dup_lo(ps);
                    uint32_t h[4];
                    e2m1x8_to_f16(words[w], h);
                    fo[w * 32 + lane] = make_uint4(f16x2_mul(h[0], sc), f16x2_mul(h[1], sc),
                                                   f16x2_mul(h[2], sc), f16x2_mul(h[3], sc));
                }
            } else {
#pragma unroll
                for (int w = 0; w < 8; ++w)
                    fo[w * 32 + lane] = make_uint4(0u, 0u, 0u, 0u);
            }
            __threadfence_block();
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(fb);  // the B fragments are in the slot
        issued = i + 1;
        cc_next(c, p);
    }
    if (lane == 0) {
        for (int64_t i = issued > kCcSlots ? issued - kCcSlots : 0; i < issued; ++i) {
            const long long t0 = clock64();
            while (!mbar_test(smem_u32(&full[i % kCcSlots]), (uint32_t)((i / kCcSlots) & 1)) &&
                   clock64() - t0 < kWaitBudget) {
            }
        }
    }
}

// A compute warp (M <= 8): rows 32 w + 16 b + g and + 8 (b = 0, 1) of every
// tile of the CTA's stream range.
// Lane (g, t) reads 16-byte chunks t and 4 + t of its two rows in the
// swizzled image (row r's chunk c at r * 128 + ((c ^ (r & 7)) << 4), and
// r & 7 = g), folds each 16-block's scale into the decoded codes (exact in
// f16) and runs two m16n8k16 MMAs per code word against the copy warp's B
// fragments (the same element order), FP32 accumulation in stage order.
__device__ void cc_consume(const TcParams& p, int64_t lo, int64_t cnt, const uint8_t* sC,
                               uint64_t* full, uint64_t* empty, volatile int* abort_flag, int w,
                               int lane)
{
    const int g = lane >> 2, t = lane & 3;
    CcCursor c;
    cc_cursor_at(c, p, lo);
    float acc[2][4], acc2[2][4];
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int q = 0; q < 4; ++q)
            acc[b][q] = acc2[b][q] = 0.f;
    for (int64_t i = 0; i < cnt; ++i) {
        const int slot = (int)(i % kCcSlots);
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&full[slot]), (uint32_t)((i / kCcSlots) & 1),
                                               abort_flag, p.status)))
            break;
        const TcItem& it = p.item[c.item];
        const uint8_t* sl = sC + slot * kCcBytes;
        const uint4* xf = reinterpret_cast<const uint4*>(sl + kCcXOff) + lane;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int ra = 32 * w + 16 * b + g, rb = ra + 8;
            const uint4 a0 = *reinterpret_cast<const uint4*>(sl + ra * 128 + ((t ^ g) << 4));
            const uint4 a1 = *reinterpret_cast<const uint4*>(sl + ra * 128 + (((4 + t) ^ g) << 4));
            const uint4 b0 = *reinterpret_cast<const uint4*>(sl + rb * 128 + ((t ^ g) << 4));
            const uint4 b1 = *reinterpret_cast<const uint4*>(sl + rb * 128 + (((4 + t) ^ g) << 4));
            const uint8_t* sa = sl + kABytes + ra * 16;
            const uint8_t* sb = sl + kABytes + rb * 16;
            const uint32_t sa01 = e4m3x2_to_f16x2_bits(*reinterpret_cast<const unsigned short*>(sa + 2 * t));
            const uint32_t sa23 = e4m3x2_to_f16x2_bits(*reinterpret_cast<const unsigned short*>(sa + 8 + 2 * t));
            const uint32_t sb01 = e4m3x2_to_f16x2_bits(*reinterpret_cast<const unsigned short*>(sb + 2 * t));
            const uint32_t sb23 = e4m3x2_to_f16x2_bits(*reinterpret_cast<const unsigned short*>(sb + 8 + 2 * t));
            const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const uint32_t wb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int wd = 0; wd < 8; ++wd) {
                const uint32_t pa = wd < 4 ? sa01 : sa23, pb = wd < 4 ? sb01 : sb23;
                const uint32_t sA = (wd & 2) ? f16x2_dup_hi(pa) : f16x2_dup_lo(pa);
                const uint32_t sB = (wd & 2) ? f16x2_dup_hi(pb) : f16x2_dup_lo(pb);
                uint32_t ha[4], hb[4];
                e2m1x8_to_f16(wa[wd], ha);
                e2m1x8_to_f16(wb[wd], hb);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    ha[q] = f16x2_mul(ha[q], sA);
                    hb[q] = f16x2_mul(hb[q], sB);
                }
                const uint4 xb = xf[wd * 32];
                mma_m16n8k16(acc[b], ha[0], hb[0], ha[1], hb[1], xb.x, xb.y);
                mma_m16n8k16(acc2[b], ha[2], hb[2], ha[3], hb[3], xb.z, xb.w);
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(&empty[slot]));
        if (c.st == c.nst - 1) {
            const float gxw = __fmul_rn(__ldg(it.xg), __ldg(it.wg));
            const OutY y = {it.y, p.y_bf16};
            const int m0 = 2 * t, m1 = m0 + 1;
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int64_t ra = (int64_t)c.tile * kRows + 32 * w + 16 * b + g, rb = ra + 8;
                const float d[4] = {acc[b][0] + acc2[b][0], acc[b][1] + acc2[b][1],
                                    acc[b][2] + acc2[b][2], acc[b][3] + acc2[b][3]};
                if (m0 < p.m) {
                    if (ra < it.n)
                        store_y(y, (int64_t)m0 * it.n + ra, d[0] * gxw);
                    if (rb < it.n)
                        store_y(y, (int64_t)m0 * it.n + rb, d[2] * gxw);
                }
                if (m1 < p.m) {
                    if (ra < it.n)
                        store_y(y, (int64_t)m1 * it.n + ra, d[1] * gxw);
                    if (rb < it.n)
                        store_y(y, (int64_t)m1 * it.n + rb, d[3] * gxw);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    acc[b][q] = acc2[b][q] = 0.f;
            }
        }
        cc_next(c, p);
    }
}

template <int NMMA, bool TILED>
__global__ void __launch_bounds__(tc_threads<NMMA, TILED>(), 1) tc_chain_kernel(const __grid_constant__ TcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kStages], aux_bar[kStages], empty_bar[kStages];
    __shared__ __align__(8) uint64_t accf_bar[2], acce_bar[2], drain_bar;
    __shared__ __align__(8) uint64_t cfull_bar[kCcSlots], cempty_bar[kCcSlots];
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;
    __shared__ int epi_fail_s;  // an epilogue warp gave up: every epilogue warp stops
    __shared__ int last_s;

    asm volatile("griddepcontrol.launch_dependents;");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t lo = p.start[blockIdx.x], hi = p.start[blockIdx.x + 1];
    const int32_t total = hi - lo;  // this CTA's stages
    // tile-aligned (1024-byte) ring: weight slots, then activation slots
    const uint32_t ring = (smem_u32(smem_raw) + 1023u) & ~1023u;
    constexpr int kBBytes = b_bytes<NMMA>();
    const uint32_t sA0 = ring, sB0 = ring + kStages * kABytes, sC0 = sB0 + kStages * kBBytes;
    uint8_t* sB_gen = smem_raw + (sB0 - smem_u32(smem_raw));
    const uint8_t* sC_gen = smem_raw + (sC0 - smem_u32(smem_raw));

    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&tmem_base_s)), "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&aux_bar[s]), 4);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&accf_bar[b]), 1);
            mbar_init(smem_u32(&acce_bar[b]), 4);
        }
        mbar_init(smem_u32(&drain_bar), 1);
        for (int s = 0; s < kCcSlots; ++s) {
            mbar_init(smem_u32(&cfull_bar[s]), 2);  // the copies, and the B fragments
            mbar_init(smem_u32(&cempty_bar[s]), kStreamWarps);
        }
        abort_s = 0;
        epi_fail_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    const uint32_t tmem = tmem_base_s;
    volatile int* abort_flag = &abort_s;

    if (warp == 0) {
        // ---- TMA producer: weight codes of every stage ----------------------------
        if (lane == 0 && total > 0) {
            Cursor c;
            cursor_at(c, p, lo);
            // L2 prefetch cursor: kL2Ahead stages ahead of the copies issued
            Cursor pc;
            cursor_at(pc, p, lo);
            auto l2_prefetch = [&](const Cursor& q) {
                if constexpr (TILED) {
                    const size_t blk = (size_t)q.tile * q.nst + q.st;
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                                 ::"l"(p.item[q.item].wq + blk * kABytes), "r"(kABytes)
                                 : "memory");
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                                 ::"l"(p.item[q.item].ws + blk * kSBytes), "r"(kSBytes)
                                 : "memory");
                } else {
                    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];"
                                 ::"l"(&p.wmap[q.item]), "r"(q.st * 128), "r"(q.tile * kRows)
                                 : "memory");
                }
            };
            int32_t pfd = 0;  // stages prefetched so far
            if constexpr (kL2Ahead > 0) {
                // the ring's first kStages stages are copied at once; prefetch the
                // ones after them up to the distance
                for (int32_t j = 0; j < kStages && j < total; ++j)
                    cursor_next_stage(pc, p);
                pfd = kStages < total ? kStages : total;
                for (; pfd < kL2Ahead && pfd < total; ++pfd) {
                    l2_prefetch(pc);
                    cursor_next_stage(pc, p);
                }
            }
            int32_t issued = 0;
            for (int32_t i = 0; i < total; ++i) {
                const int slot = i % kStages;
                if (i >= kStages &&
                    !mbar_wait(smem_u32(&empty_bar[slot]), ((i / kStages) - 1) & 1, abort_flag,
                               p.status))
                    break;
                const uint32_t fb = smem_u32(&full_bar[slot]);
                if constexpr (TILED) {
                    // tile-major layout: the stage's codes, already in the swizzled
                    // shared-memory image, are one contiguous 16 KB block (its
                    // scales go through the scale warps' registers)
                    const size_t blk = (size_t)c.tile * c.nst + c.st;
                    mbar_expect_tx(fb, kABytes);
                    asm volatile(
                        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
                        "[%0], [%1], %2, [%3];" ::"r"(sA0 + slot * kABytes),
                        "l"(p.item[c.item].wq + blk * kABytes), "r"(kABytes), "r"(fb)
                        : "memory");
                } else {
                    mbar_expect_tx(fb, kABytes);
                    asm volatile(
                        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::"
                        "bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(sA0 + slot * kABytes),
                        "l"(&p.wmap[c.item]), "r"(c.st * 128), "r"(c.tile * kRows), "r"(fb)
                        : "memory");
                }
                issued = i + 1;
                cursor_next_stage(c, p);
                if constexpr (kL2Ahead > 0) {
                    if (pfd < total && pfd <= i + kL2Ahead) {
                        l2_prefetch(pc);
                        cursor_next_stage(pc, p);
                        ++pfd;
                    }
                }
            }
            // drain: every copy issued has landed before the CTA can exit
            for (int32_t i = issued > kStages ? issued - kStages : 0; i < issued; ++i) {
                const long long t0 = clock64();
                while (!mbar_test(smem_u32(&full_bar[i % kStages]), (i / kStages) & 1) &&
                       clock64() - t0 < kWaitBudget) {
                }
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer: one accumulator per tile segment --------------------------------
        if (lane == 0 && total > 0) {
            Cursor c;
            cursor_at(c, p, lo);
            const uint32_t idesc = instr_desc(NMMA);
            int32_t i = 0, tcount = 0;
            bool ok = true;
            while (ok && i < total) {
                const int buf = tcount & 1;
                if (tcount >= 2 && !mbar_wait(smem_u32(&acce_bar[buf]), ((tcount >> 1) - 1) & 1,
                                              abort_flag, p.status))
                    break;
                asm volatile("tcgen05.fence::after_thread_sync;");
                const uint32_t dcol = tmem + (uint32_t)(buf * 32);
                const int32_t len = c.nst - c.st < total - i ? c.nst - c.st : total - i;
                for (int32_t s = 0; s < len; ++s, ++i) {
                    const int slot = i % kStages;
                    const uint32_t ph = (i / kStages) & 1;
                    if (!mbar_wait(smem_u32(&full_bar[slot]), ph, abort_flag, p.status) ||
                        !mbar_wait(smem_u32(&aux_bar[slot]), ph, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;");
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint64_t ad = operand_desc(sA0 + slot * kABytes + 32 * j);
                        const uint64_t bd = operand_desc(sB0 + slot * kBBytes + 32 * j);
                        const uint32_t sfa = tmem + kColSfa + slot * 16 + 4 * j;
                        const uint32_t sfb = tmem + kColSfb + slot * 16 + 4 * j;
                        asm volatile(
                            "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %6, 0;\n\t"
                            "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X "
                            "[%0], %1, %2, %3, [%4], [%5], q;\n\t}" ::"r"(dcol),
                            "l"(ad), "l"(bd), "r"(idesc), "r"(sfa), "r"(sfb), "r"(s | j)
                            : "memory");
                    }
                    asm volatile(
                        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
                        "[%0];" ::"r"(smem_u32(&empty_bar[slot]))
                        : "memory");
                }
                if (!ok)
                    break;
                asm volatile(
                    "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                    ::"r"(smem_u32(&accf_bar[buf]))
                    : "memory");
                ++tcount;
                cursor_next_tile(c, p);
            }
            // drain: every MMA issued has completed before tensor memory is freed
            asm volatile(
                "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                ::"r"(smem_u32(&drain_bar))
                : "memory");
            const long long t0 = clock64();
            while (!mbar_test(smem_u32(&drain_bar), 0) && clock64() - t0 < kWaitBudget) {
            }
        }
    } else if (warp < 6) {
        // ---- block scales and activation codes of every stage --------------------------
        asm volatile("griddepcontrol.wait;" ::: "memory");  // x_q / x_s come from the producer
        const int q = warp & 3;               // tensor-memory lane quarter of this warp
        const int r = 32 * q + lane;          // weight row within the tile
        const int u = (warp - 2) * 32 + lane;  // activation code chunk (row u / 8, 16 bytes u % 8)
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        if (total > 0) {
            Cursor pf;
            cursor_at(pf, p, lo);
            AuxLoad ring[kPrefetch];
#pragma unroll
            for (int d = 0; d < kPrefetch; ++d) {
                if (d < total) {
                    aux_load<NMMA, TILED>(ring[d], p, pf, r, lane, u);
                    cursor_next_stage(pf, p);
                }
            }
            bool ok = true;
            for (int32_t i0 = 0; ok && i0 < total; i0 += kPrefetch) {
#pragma unroll
                for (int d = 0; d < kPrefetch; ++d) {
                    const int32_t i = i0 + d;
                    if (i >= total)
                        break;
                    const int slot = i % kStages;
                    // warp-uniform decision: the tcgen05 stores below are .sync.aligned
                    if (i >= kStages &&
                        !__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&empty_bar[slot]),
                                                           ((i / kStages) - 1) & 1, abort_flag,
                                                           p.status))) {
                        ok = false;
                        break;
                    }
                    const uint4 sa4 = ring[d].sa;
                    asm volatile("tcgen05.fence::after_thread_sync;");
                    const uint32_t sa[4] = {sa4.x, sa4.y, sa4.z, sa4.w};
                    const uint32_t sb[4] = {ring[d].sb.x, ring[d].sb.y, ring[d].sb.z, ring[d].sb.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        tmem_st1(lane_base + kColSfa + slot * 16 + 4 * j + q, sa[j]);
                        tmem_st1(lane_base + kColSfb + slot * 16 + 4 * j, sb[j]);
                    }
                    // activation codes in the swizzled layout TMA would write
                    uint8_t* bs = sB_gen + slot * kBBytes;
                    if (u < p.m * 8) {
                        const int n = u >> 3, ch = u & 7;
                        *reinterpret_cast<uint4*>(bs + n * 128 + ((ch ^ (n & 7)) << 4)) = ring[d].b0;
                    }
                    if constexpr (NMMA > 16) {
                        if (u + 128 < p.m * 8) {
                            const int n = (u + 128) >> 3, ch = (u + 128) & 7;
                            *reinterpret_cast<uint4*>(bs + n * 128 + ((ch ^ (n & 7)) << 4)) =
                                ring[d].b1;
                        }
                    }
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    asm volatile("tcgen05.fence::before_thread_sync;");
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(smem_u32(&aux_bar[slot]));
                    if (i + kPrefetch < total) {
                        aux_load<NMMA, TILED>(ring[d], p, pf, r, lane, u);
                        cursor_next_stage(pf, p);
                    }
                }
            }
        }
    } else if (warp < kThreads / 32) {
        // ---- epilogue ----------------------------------------------------------------------
        asm volatile("griddepcontrol.wait;" ::: "memory");  // Y may still be read before
        const int q = warp & 3;
        const int r = 32 * q + lane;
        const int et = threadIdx.x - 6 * 32;  // 0..127 among the epilogue threads
        if (total > 0) {
            Cursor c;
            cursor_at(c, p, lo);
            int32_t i = 0, tcount = 0;
            while (i < total) {
                const int buf = tcount & 1;
                const int32_t st_a = c.st;
                const int32_t len = c.nst - c.st < total - i ? c.nst - c.st : total - i;
                // one decision for the four epilogue warps (they share a named
                // barrier below, so none may leave alone)
                const bool wok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&accf_bar[buf]),
                                                                   (tcount >> 1) & 1, abort_flag,
                                                                   p.status));
                if (lane == 0 && !wok)
                    epi_fail_s = 1;
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (*(volatile int*)&epi_fail_s)
                    break;
                asm volatile("tcgen05.fence::after_thread_sync;");
                uint32_t v[NMMA];
                const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * 32);
                if constexpr (NMMA == 16) {
                    asm volatile(
                        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,"
                        "%10,%11,%12,%13,%14,%15}, [%16];"
                        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                          "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
                          "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                        : "r"(taddr));
                } else {
                    asm volatile(
                        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,"
                        "%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,"
                        "%28,%29,%30,%31}, [%32];"
                        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                          "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
                          "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
                          "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
                          "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]),
                          "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                        : "r"(taddr));
                }
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                asm volatile("tcgen05.fence::before_thread_sync;");
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&acce_bar[buf]));
                const TcItem& it = p.item[c.item];
                const int64_t row = (int64_t)c.tile * kRows + r;
                const float gxw = __fmul_rn(__ldg(it.xg), __ldg(it.wg));
                const OutY y = {it.y, p.y_bf16};
                if (st_a == 0 && len == c.nst) {
                    // the whole tile's K in this accumulator
                    if (row < it.n) {
#pragma unroll
                        for (int n = 0; n < NMMA; ++n)
                            if (n < p.m)
                                store_y(y, (int64_t)n * it.n + row, __uint_as_float(v[n]) * gxw);
                    }
                } else {
                    // a tile split between CTAs: this CTA's partial into its slot (0: the
                    // tile its range starts in, 1: the tile it ends in), then the last of
                    // the tile's CTAs to arrive sums every partial in stage order
                    const int32_t T0 = it.s0 + c.tile * c.nst;  // the tile's first stage
                    float* mine = p.part + ((size_t)(2 * blockIdx.x + (lo >= T0 ? 0 : 1)) * 32) * kRows;
#pragma unroll
                    for (int n = 0; n < NMMA; ++n)
                        if (n < p.m)
                            __stcg(mine + n * kRows + r, __uint_as_float(v[n]));
                    __threadfence();
                    asm volatile("bar.sync 1, 128;" ::: "memory");
                    const int bf = cta_of_stage(p, T0), bl = cta_of_stage(p, T0 + c.nst - 1);
                    if (et == 0) {
                        const unsigned prev = atomicAdd(p.count + bf, 1u);
                        last_s = prev == (unsigned)(bl - bf);
                    }
                    asm volatile("bar.sync 1, 128;" ::: "memory");
                    if (last_s) {
                        __threadfence();
                        float acc[NMMA];
#pragma unroll
                        for (int n = 0; n < NMMA; ++n)
                            acc[n] = 0.0f;
                        // partials in stage order, two contributors' loads in flight
                        // at a time (the additions keep that order)
                        for (int cc = bf; cc <= bl; cc += 2) {
                            const bool two = cc + 1 <= bl;
                            const float* s0 =
                                p.part + ((size_t)(2 * cc + (p.start[cc] >= T0 ? 0 : 1)) * 32) * kRows;
                            const float* s1 =
                                two ? p.part + ((size_t)(2 * (cc + 1) +
                                                         (p.start[cc + 1] >= T0 ? 0 : 1)) * 32) * kRows
                                    : s0;
                            float a0[NMMA], a1[NMMA];
#pragma unroll
                            for (int n = 0; n < NMMA; ++n) {
                                if (n < p.m) {
                                    a0[n] = __ldcg(s0 + n * kRows + r);
                                    a1[n] = two ? __ldcg(s1 + n * kRows + r) : 0.0f;
                                }
                            }
#pragma unroll
                            for (int n = 0; n < NMMA; ++n) {
                                if (n < p.m) {
                                    acc[n] += a0[n];
                                    if (two)
                                        acc[n] += a1[n];
                                }
                            }
                        }
                        if (row < it.n) {
#pragma unroll
                            for (int n = 0; n < NMMA; ++n)
                                if (n < p.m)
                                    store_y(y, (int64_t)n * it.n + row, acc[n] * gxw);
                        }
                        if (et == 0)
                            atomicExch(p.count + bf, 0u);
                    }
                }
                i += len;
                ++tcount;
                cursor_next_tile(c, p);
            }
        }
    } else if constexpr (has_stream<NMMA, TILED>()) {
        // ---- stream warps: the last tiles of every linear on mma.sync -------------------
        const int w = warp - kThreads / 32;  // compute warps 0 .. kStreamWarps - 1, then the copy warp
        const int64_t all = cc_boundary(p, INT64_MAX);
        const int64_t lo = cc_boundary(p, all * blockIdx.x / gridDim.x);
        const int64_t cnt = cc_boundary(p, all * (blockIdx.x + 1) / gridDim.x) - lo;
        if (cnt > 0 && p.m <= 8) {
            if (w == kStreamWarps) {
                cc_produce(p, lo, cnt, sC0, smem_raw + (sC0 - smem_u32(smem_raw)), cfull_bar,
                           cempty_bar, abort_flag, lane);
            } else {
                asm volatile("griddepcontrol.wait;" ::: "memory");  // x_q / x_s come from the producer
                cc_consume(p, lo, cnt, sC_gen, cfull_bar, cempty_bar, abort_flag, w, lane);
            }
        }
    }

    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols));
}

// ---- host side ---------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// Weight codes [n][k/2] as a 2-D tensor of bytes: boxes of 128 bytes x 128
// rows with 128-byte swizzle (rows past n read as zeros).
bool weight_map(CUtensorMap* m, const uint8_t* wq, int64_t n, int64_t k)
{
    auto enc = tensor_map_encoder();
    if (enc == nullptr)
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)(k / 2), (cuuint64_t)n};
    const cuuint64_t strides[1] = {(cuuint64_t)(k / 2)};
    const cuuint32_t box[2] = {128, kRows};
    const cuuint32_t es[2] = {1, 1};
#ifndef NVFP4_TC_L2_PROMOTION
#define NVFP4_TC_L2_PROMOTION CU_TENSOR_MAP_L2_PROMOTION_L2_256B
#endif
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(wq), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, NVFP4_TC_L2_PROMOTION,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NMMA, bool TILED>
cudaError_t launch_tc_t(TcParams& prm, int grid, cudaStream_t stream, bool pdl)
{
    auto kern = tc_chain_kernel<NMMA, TILED>;
    const int dev = current_device();
    const size_t smem = smem_bytes<NMMA, TILED>();
    cudaError_t e = ensure_smem_limit(kern, smem, dev);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(tc_threads<NMMA, TILED>(), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, prm);
}

}  // namespace

bool tc_shape_ok(int64_t m, int64_t n, int64_t k)
{
    return m >= 1 && m <= 32 && n >= 1 && n < (int64_t(1) << 30) && k >= kStageK &&
           k % kStageK == 0 && k < (int64_t(1) << 30);
}

int64_t tc_workspace_bytes()
{
    int grid = device_sm_count(current_device());
    if (grid > kTcMaxCtas)
        grid = kTcMaxCtas;
    return 1024 + (int64_t)2 * grid * 32 * kRows * (int64_t)sizeof(float);
}

cudaError_t launch_tc_chain(const ChainLinear* items, int count, int m, bool quantize, bool x_bf16,
                            bool y_bf16, cudaStream_t stream, bool pdl, void* workspace,
                            int64_t workspace_bytes, bool tiled)
{
    if (count < 1 || count > kTcMaxItems || m < 1 || m > 32)
        return cudaErrorInvalidValue;
    static thread_local TcParams prm;  // 31 KB: kept off the stack
    prm.count_items = count;
    prm.m = m;
    prm.y_bf16 = y_bf16 ? 1 : 0;
    cudaError_t e = device_status_address(&prm.status);
    if (e != cudaSuccess)
        return e;
    // at M <= 8, with tile-major weights, the stream warps take the last tiles
    // of every linear (a share of its tiles, at least one left to the tensor
    // cores)
    const bool rows_to_stream = m <= 8 && tiled;
    const int64_t share = rows_to_stream ? kStreamShare[m] : 0;
    int64_t stages = 0;
    for (int i = 0; i < count; ++i) {
        const ChainLinear& L = items[i];
        TcItem& it = prm.item[i];
        if (!tiled && !weight_map(&prm.wmap[i], L.wq, L.n, L.k))
            return cudaErrorInvalidValue;
        it.wq = L.wq;
        it.xq = L.xq;
        it.xs = L.xs;
        it.xg = L.xg;
        it.ws = L.ws;
        it.wg = L.wg;
        it.y = L.y;
        it.n = (int32_t)L.n;
        it.k = (int32_t)L.k;
        it.s0 = (int32_t)stages;
        const int64_t tiles = (L.n + kRows - 1) / kRows;
        int64_t cc = 0;
        if (rows_to_stream) {
            cc = (tiles * share + 500) / 1000;
            if (cc > tiles - 1)
                cc = tiles - 1;
        }
        it.ttiles = (int32_t)(tiles - cc);
        stages += (tiles - cc) * (L.k / kStageK);
    }
    if (stages >= (int64_t(1) << 31))
        return cudaErrorInvalidValue;
    const int dev = current_device();
    int grid = device_sm_count(dev);
    if (grid > kTcMaxCtas)
        grid = kTcMaxCtas;
    // every stage moves the same weight bytes (16 KB of codes, 2 KB of scales)
    const bool streamk = workspace != nullptr && workspace_bytes >= tc_workspace_bytes();
    if (streamk) {
        // stage ranges of equal length; tiles cut at a range boundary are
        // combined through the workspace
        if (grid > stages)
            grid = (int)stages;
        for (int b = 0; b <= grid; ++b)
            prm.start[b] = (int32_t)(stages * b / grid);
        prm.count = static_cast<unsigned*>(workspace);
        prm.part = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + 1024);
    } else {
        // ranges on tile boundaries, each near an equal share of the stages
        int64_t tiles = 0;
        for (int i = 0; i < count; ++i)
            tiles += prm.item[i].ttiles;
        if (grid > tiles)
            grid = (int)tiles;
        int i = 0;
        for (int b = 0; b <= grid; ++b) {
            const int64_t target = stages * b / grid;
            // first tile boundary at or after target
            while (i < count - 1 &&
                   prm.item[i + 1].s0 <= target) {
                ++i;
            }
            const int64_t nst = prm.item[i].k / kStageK;
            const int64_t ti = (target - prm.item[i].s0 + nst - 1) / nst;
            const int64_t g = prm.item[i].s0 + ti * nst;
            prm.start[b] = (int32_t)(g < stages ? g : stages);
        }
        prm.start[0] = 0;
        prm.start[grid] = (int32_t)stages;
        for (int b = 1; b <= grid; ++b)
            if (prm.start[b] < prm.start[b - 1])
                prm.start[b] = prm.start[b - 1];
        prm.count = nullptr;
        prm.part = nullptr;
    }
    prm.grid = grid;

    bool tc_pdl = pdl;
    if (quantize) {
        e = launch_chain_quant(items, count, m, x_bf16, stream, pdl);
        if (e != cudaSuccess)
            return e;
        tc_pdl = true;  // the weight loads do not depend on the quantiser
    }
    if (tiled)
        return m <= 16 ? launch_tc_t<16, true>(prm, grid, stream, tc_pdl)
                       : launch_tc_t<32, true>(prm, grid, stream, tc_pdl);
    return m <= 16 ? launch_tc_t<16, false>(prm, grid, stream, tc_pdl)
                   : launch_tc_t<32, false>(prm, grid, stream, tc_pdl);
}

cudaError_t launch_gemm_tc(const GemmArgs& a, bool pdl, void* workspace, int64_t workspace_bytes,
                           bool tiled)
{
    const ChainLinear one = {nullptr, a.xg, const_cast<uint8_t*>(a.xq), const_cast<uint8_t*>(a.xs),
                             a.wq, a.ws, a.wg, a.y.p, a.n, a.k};
    return launch_tc_chain(&one, 1, a.m, false, false, a.y.bf16 != 0, a.stream, pdl, workspace,
                           workspace_bytes, tiled);
}

// ---- tile-major weight layout ---------------------------------------------------

namespace {

// One 16-byte chunk of codes per thread: padded row p (tile p / 128, row
// r = p % 128), chunk h of the row (stage h / 8, chunk c = h % 8 of the
// stage's 128 bytes) goes to block (tile, stage), row r, swizzled chunk
// c ^ (r % 8) -- the image TMA with 128-byte swizzle writes to shared memory.
// Rows past n are zero.
__global__ void tile_codes_kernel(const uint8_t* __restrict__ wq, int64_t n, int64_t k,
                                  int64_t rows_padded, uint8_t* __restrict__ tq)
{
    const int64_t chunks = k / 32;  // 16-byte chunks per row
    const int64_t total = rows_padded * chunks;
    const int64_t nst = k / kStageK;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = i / chunks, h = i - row * chunks;
        const int64_t t = row / kRows, r = row - t * kRows, st = h / 8, c = h - st * 8;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < n)
            v = __ldg(reinterpret_cast<const uint4*>(wq + row * (k / 2)) + h);
        *reinterpret_cast<uint4*>(tq + ((t * nst + st) * kRows + r) * 128 + ((c ^ (r & 7)) << 4)) = v;
    }
}

// One stage's 16 scale bytes of one padded row per thread: block (tile, stage),
// row r at 16 r.  Rows past n are zero.
__global__ void tile_scales_kernel(const uint8_t* __restrict__ ws, int64_t n, int64_t k,
                                   int64_t rows_padded, uint8_t* __restrict__ ts)
{
    const int64_t nst = k / kStageK;
    const int64_t total = rows_padded * nst;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = i / nst, st = i - row * nst;
        const int64_t t = row / kRows, r = row - t * kRows;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < n)
            v = __ldg(reinterpret_cast<const uint4*>(ws + row * (k / 16)) + st);
        *reinterpret_cast<uint4*>(ts + ((t * nst + st) * kRows + r) * 16) = v;
    }
}

}  // namespace

int64_t tiled_code_bytes(int64_t n, int64_t k)
{
    return (n + kRows - 1) / kRows * kRows * (k / 2);
}

int64_t tiled_scale_bytes(int64_t n, int64_t k)
{
    return (n + kRows - 1) / kRows * kRows * (k / 16);
}

cudaError_t launch_tile_weight(const uint8_t* wq, const uint8_t* ws, int64_t n, int64_t k,
                               uint8_t* tq, uint8_t* ts, cudaStream_t stream)
{
    const int64_t rows = (n + kRows - 1) / kRows * kRows;
    const int sms = device_sm_count(current_device());
    const int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 8;
    int64_t g1 = (rows * (k / 32) + 255) / 256, g2 = (rows * (k / kStageK) + 255) / 256;
    g1 = g1 < 1 ? 1 : (g1 > cap ? cap : g1);
    g2 = g2 < 1 ? 1 : (g2 > cap ? cap : g2);
    tile_codes_kernel<<<(unsigned)g1, 256, 0, stream>>>(wq, n, k, rows, tq);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    tile_scales_kernel<<<(unsigned)g2, 256, 0, stream>>>(ws, n, k, rows, ts);
    return cudaGetLastError();
}

}  // namespace nvfp4
