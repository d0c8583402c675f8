// ptx.cuh -- inline-PTX wrappers for sm_103a: mbarriers, TMA tensor loads,
// timers and the bounded wait used by every kernel of the library.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "../../include/dep_projection.h"

namespace dep {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier ----
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the phase with the given parity has completed, for at most
// limit_ns nanoseconds.  Returns false if it gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (globaltimer_ns() - t0 > limit_ns)
            return false;
    }
}

// ---- TMA (bulk tensor copies, global -> shared, completion on an mbarrier) ----
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int32_t c0,
                                            int32_t c1, uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
        : "memory");
}

// Three-dimensional form (maps of encode_bf16_3d_blocks: c0 = 0, c1 = row,
// c2 = first 64-column block).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int32_t c0, int32_t c1,
                                            int32_t c2, uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// L2 policies: streamed-once data (the weight) and reused data (activations).
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---- programmatic dependent launch ----
// Let the next grid in the stream be scheduled once every block of this grid has
// issued this (no-op when the launch did not allow it).
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Wait until the preceding grid in the stream has completed and its memory is
// visible (returns at once when there is no programmatic dependency).
__device__ __forceinline__ void griddep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Record the first nonzero code in the device status word.
__device__ __forceinline__ void record_status(int *status, int code)
{
    if (status)
        atomicCAS(status, 0, code);
}

// Bounds check of the DEP_DEBUG build: an index at or past the buffer's size
// records DEP_DEV_BOUNDS and the caller skips the access.  In other builds the
// check is compiled away (always true).
__device__ __forceinline__ bool dbg_ok(unsigned long long idx, unsigned long long n, int *status)
{
#ifdef DEP_DEBUG
    if (idx < n)
        return true;
    record_status(status, DEP_DEV_BOUNDS);
    return false;
#else
    (void)idx;
    (void)n;
    (void)status;
    return true;
#endif
}
// The same for a range [off, off + len).
__device__ __forceinline__ bool dbg_range(unsigned long long off, unsigned long long len, unsigned long long n,
                                          int *status)
{
    return dbg_ok(off + len - 1, n, status) && dbg_ok(off, n, status);
}

// ---- tcgen05 (5th-generation tensor cores, accumulators in tensor memory) ----
namespace tc {

// Allocate ncols (a power of two >= 32) TMEM columns; the address lands in shared
// memory at dst.  Executed by one whole warp.
__device__ __forceinline__ void alloc(uint32_t dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, BF16 inputs, FP32 accumulation.
__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on an mbarrier when every tcgen05 op issued so far by this thread completes.
__device__ __forceinline__ void commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns per thread.
__device__ __forceinline__ void ld16(uint32_t taddr, uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
        "%12, %13, %14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}
__device__ __forceinline__ void wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand tile in the 128-byte swizzle
// layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B (rows of 128 bytes, groups of
// 8 rows 1024 bytes apart).  Fields: start address >> 4 (bits 0-13), leading
// byte offset >> 4 (16-29, unused for this layout: 1), stride byte offset >> 4
// (32-45: 1024 B), descriptor version 1 (46-47), base offset 0 (49-51),
// swizzle mode 2 = 128 B (61-63).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr)
{
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16: FP32 accumulator (bits 4-5 = 1), A and B
// BF16 (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 in
// bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Issue H consecutive 16-column K steps of one stage into accumulator d, fully
// unrolled with constant descriptor offsets: step i reads slice i / 4 (A at
// ad + i / 4 slices of A_BYTES, B likewise) at K offset 16 (i % 4) inside the
// slice's 128-byte rows (2 descriptor units of 16 bytes per step).  ad and bd
// are the descriptors of the first step.  One thread issues a tcgen05.mma only
// every ~45 cycles at best, and address arithmetic between the instructions
// adds to that, so the loop carries none.
template <int H, int A_BYTES, int B_BYTES>
__device__ __forceinline__ void mma_steps(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t &accumulate)
{
#pragma unroll
    for (int i = 0; i < H; ++i) {
        const uint64_t ka = (uint64_t)(((i / 4) * A_BYTES) >> 4) + 2 * (i % 4);
        const uint64_t kb = (uint64_t)(((i / 4) * B_BYTES) >> 4) + 2 * (i % 4);
        mma_bf16(d, ad + ka, bd + kb, idesc, accumulate);
        accumulate = 1;
    }
}

// The K steps [k0, k0 + n) of a stage whose slices start at a0 (A) and b0 (B),
// n in {2, 4, 8, 16}; k0 % 4 == 0 unless n == 2 (then the steps stay in one slice).
template <int A_BYTES, int B_BYTES>
__device__ __forceinline__ void mma_stage(uint32_t d, uint32_t a0, uint32_t b0, int k0, int n, uint32_t idesc,
                                          uint32_t &accumulate)
{
    const uint64_t ad = desc_sw128(a0 + (uint32_t)((k0 / 4) * A_BYTES)) + 2 * (k0 % 4);
    const uint64_t bd = desc_sw128(b0 + (uint32_t)((k0 / 4) * B_BYTES)) + 2 * (k0 % 4);
    switch (n) {
    case 16: mma_steps<16, A_BYTES, B_BYTES>(d, ad, bd, idesc, accumulate); break;
    case 8: mma_steps<8, A_BYTES, B_BYTES>(d, ad, bd, idesc, accumulate); break;
    case 4: mma_steps<4, A_BYTES, B_BYTES>(d, ad, bd, idesc, accumulate); break;
    default: mma_steps<2, A_BYTES, B_BYTES>(d, ad, bd, idesc, accumulate); break;
    }
}

}  // namespace tc

}  // namespace dep
