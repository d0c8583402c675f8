// probe.cu -- read-only streaming ceiling of the device's memory.
//
// The projection reads each weight once and writes almost nothing, so the
// fraction of the device's bandwidth it reaches is best judged against a
// kernel that only reads: a plain copy also writes as many bytes as it reads.
// Every thread keeps four 16-byte loads in flight (non-coherent path, no L1
// allocation), folds the words into an XOR, and each warp
// XORs its result into one word so that no load can be dropped.  Grid: four
// blocks of 512 threads per SM.
#include "internal.h"

namespace dep {
namespace {

constexpr int kProbeThreads = 512;

__device__ __forceinline__ uint4 ld_stream(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__global__ void __launch_bounds__(kProbeThreads)
    read_probe_kernel(const uint4 *__restrict__ p, size_t n, unsigned long long *__restrict__ sink)
{
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    uint32_t acc = 0;
    for (; i + 3 * stride < n; i += 4 * stride) {
        const uint4 a = ld_stream(p + i), b = ld_stream(p + i + stride), c = ld_stream(p + i + 2 * stride),
                    d = ld_stream(p + i + 3 * stride);
        acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
    }
    for (; i < n; i += stride) {
        const uint4 a = ld_stream(p + i);
        acc ^= a.x ^ a.y ^ a.z ^ a.w;
    }
    for (int off = 16; off > 0; off >>= 1)
        acc ^= __shfl_xor_sync(0xffffffffu, acc, off);
    if ((threadIdx.x & 31) == 0)
        atomicXor(sink, (unsigned long long)acc);
}

}  // namespace
}  // namespace dep

extern "C" dep_status_t dep_projection_probe_read(const void *p, size_t bytes, void *sink, void *stream)
{
    if (!p || !sink || bytes == 0)
        return DEP_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(p) & 15u) || (bytes & 15u) || (reinterpret_cast<uintptr_t>(sink) & 7u))
        return DEP_ERR_MISALIGNED;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess) {
        cudaGetLastError();
        return DEP_ERR_CUDA;
    }
    dep::read_probe_kernel<<<sms * 4, dep::kProbeThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4 *>(p), bytes / 16, static_cast<unsigned long long *>(sink));
    if (cudaGetLastError() != cudaSuccess)
        return DEP_ERR_CUDA;
    return DEP_OK;
}
