// staging.cu -- zero-copy staging of x and y for the host-buffer entry point.
//
// When the caller's host buffers are pinned (mapped into the device's address
// space), x is gathered into the plan's device staging area by a small kernel
// instead of a memcpy; the projection stores y into the mapped buffer itself,
// or (the cluster and x-on-M kinds, whose y stores are not rows of contiguous
// bytes across a warp) writes the staging area and the same kernel copies y
// back.  Chained by programmatic
// dependent launch: each copy triggers its dependents at once and waits for
// the preceding grid before it reads (so a source written by earlier work in
// the stream is complete, and the staging area is no longer read by an earlier
// projection); the projection kernel launches early and streams its first
// weight stages while x is still arriving (it reads x only after its
// griddepcontrol.wait); the next call's gather launches early the same way, so
// no launch gap separates the calls.  Plain loads and stores of mapped host
// memory; 16-byte vectors where both sides allow it, 2-byte elements for the
// rest.
#include "internal.h"
#include "ptx.cuh"

namespace dep {
namespace {

constexpr int kStageThreads = 256;

__global__ void __launch_bounds__(kStageThreads)
    stage_copy_kernel(const uint16_t *__restrict__ src, uint16_t *__restrict__ dst, size_t n, int wait_first)
{
    if (wait_first)
        griddep_wait();  // the source is written by the preceding grid
    griddep_launch_dependents();
    const size_t tid = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    const size_t nv = n / 8;  // 16-byte vectors (both pointers are 16-byte aligned)
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
    // Four loads in flight per thread before their stores: reads of mapped host
    // memory take microseconds.
    size_t i = tid;
    for (; i + 3 * stride < nv; i += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            v[u] = s4[i + u * stride];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            d4[i + u * stride] = v[u];
    }
    for (; i < nv; i += stride)
        d4[i] = s4[i];
    for (size_t j = nv * 8 + tid; j < n; j += stride)
        dst[j] = src[j];
}

int copy_grid(size_t n)
{
    const size_t vecs = (n + 7) / 8;
    const size_t blocks = (vecs + kStageThreads - 1) / kStageThreads;
    return (int)(blocks < 1 ? 1 : blocks > 608 ? 608 : blocks);
}

}  // namespace

cudaError_t stage_copy(const uint16_t *src, uint16_t *dst, size_t n, bool after_preceding, cudaStream_t stream)
{
    // With after_preceding the copy is launched with the programmatic attribute
    // and waits for the preceding grid itself (a preceding kernel that does not
    // trigger its dependents, or a copy, still orders it as a plain launch
    // would); without, it is an ordinary launch.
    return launch(stage_copy_kernel, dim3(copy_grid(n)), dim3(kStageThreads), 0, stream, after_preceding, src, dst,
                  n, after_preceding ? 1 : 0);
}

}  // namespace dep
