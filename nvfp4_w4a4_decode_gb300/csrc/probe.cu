// probe.cu -- a read-only streaming kernel: the DRAM read rate that a plain
// stream of 128-bit loads reaches on this device.  It is a measurement aid
// beside the GEMM (the GEMM's weight stream is read-only too, so this is the
// ceiling its loads could reach on the same device, next to the copy peak),
// not a step of the method.
//
// Every 16-byte word of the buffer is loaded exactly once (non-allocating in
// L1, four independent loads in flight per thread) and XOR-folded, as two
// 64-bit halves, into one word per warp, which goes to the sink with one
// atomic XOR: the sink ends as the XOR of all 8-byte words of the buffer, so
// that no load can be dropped and a test can check the result.
#include "kernels.cuh"
#include "launch_cache.cuh"

namespace nvfp4 {

namespace {

constexpr int kProbeThreads = 512;
constexpr int kProbeCtasPerSm = 4;

__device__ __forceinline__ uint4 ld_probe(const uint4* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ unsigned long long fold(const uint4& v)
{
    const unsigned long long lo = ((unsigned long long)v.y << 32) | v.x;
    const unsigned long long hi = ((unsigned long long)v.w << 32) | v.z;
    return lo ^ hi;
}

__global__ void __launch_bounds__(kProbeThreads, kProbeCtasPerSm)
    read_probe_kernel(const uint4* __restrict__ buf, int64_t words, unsigned long long* sink)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    unsigned long long acc = 0ull;
    for (; w + 3 * stride < words; w += 4 * stride) {
        const uint4 a = ld_probe(buf + w);
        const uint4 b = ld_probe(buf + w + stride);
        const uint4 c = ld_probe(buf + w + 2 * stride);
        const uint4 d = ld_probe(buf + w + 3 * stride);
        acc ^= fold(a) ^ fold(b) ^ fold(c) ^ fold(d);
    }
    for (; w < words; w += stride)
        acc ^= fold(ld_probe(buf + w));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        acc ^= __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if ((threadIdx.x & 31) == 0 && acc != 0ull)
        atomicXor(sink, acc);
}

}  // namespace

cudaError_t launch_read_probe(const void* buf, int64_t bytes, unsigned long long* sink,
                              cudaStream_t stream)
{
    cudaError_t e = cudaMemsetAsync(sink, 0, sizeof(unsigned long long), stream);
    if (e != cudaSuccess || bytes == 0)
        return e;
    const int64_t words = bytes / 16;
    int64_t grid = (int64_t)device_sm_count(current_device()) * kProbeCtasPerSm;
    const int64_t need = (words + kProbeThreads - 1) / kProbeThreads;
    if (grid > need)
        grid = need;
    read_probe_kernel<<<(unsigned)grid, kProbeThreads, 0, stream>>>(
        static_cast<const uint4*>(buf), words, sink);
    return cudaGetLastError();
}

}  // namespace nvfp4
