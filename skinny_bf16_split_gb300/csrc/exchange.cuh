// exchange.cuh -- split-K partials exchanged through flagged 64-bit words.
//
// One word per (tile, piece, batch column, row): the FP32 partial in the low
// 32 bits and a "full" flag in the high 32 bits, written with one relaxed
// GPU-scope 64-bit store (single-copy atomic for an aligned word, so a reader
// that sees the flag also sees the value: no fence and no counter needed).  The
// reducing block polls the words of the other pieces (bounded in time), adds
// them in piece order with its own piece last, and clears the flags for the
// next launch (the values are kept for inspection).  Used by the tensor-core
// kernels; the region is the plan's, zeroed at allocation and never written by
// any other kernel.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace dep {
namespace xch {

constexpr unsigned long long kFull = 1ull << 32;

__device__ __forceinline__ unsigned long long load(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void store(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Publish 16 batch columns of one row: word j at p + j * col_stride, for j < ncols.
__device__ __forceinline__ void publish16(unsigned long long *p, int64_t col_stride, const uint32_t (&v)[16],
                                          int ncols)
{
#pragma unroll
    for (int j = 0; j < 16; ++j)
        if (j < ncols)
            store(p + j * col_stride, kFull | v[j]);
}

// Reduce 16 batch columns of one row: out[j] = ((p_0 + p_1) + ...) + own[j] in
// FP32, where p_i is read from piece i's word at base + i * piece_stride +
// j * col_stride (i < np, j < ncols), waiting for its flag at most limit_ns.
// Own values are kept (flag clear) at own_word + j * col_stride.  PB pieces'
// words are in flight at a time (one L2 round trip per PB pieces once they are
// published).  Returns false if a wait gave up (out is then incomplete).
template <int PB = 2>
__device__ __forceinline__ bool reduce16(unsigned long long *base, int64_t piece_stride, int64_t col_stride,
                                         int np, int ncols, const uint32_t (&own)[16],
                                         unsigned long long *own_word, float (&out)[16], uint64_t limit_ns)
{
#pragma unroll
    for (int j = 0; j < 16; ++j)
        if (j < ncols)
            store(own_word + j * col_stride, (unsigned long long)own[j]);
    bool ok = true;
    for (int p0 = 0; p0 < np; p0 += PB) {
        unsigned long long w[PB][16];
        unsigned long long *src[PB];
#pragma unroll
        for (int i = 0; i < PB; ++i) {
            src[i] = base + (int64_t)(p0 + i) * piece_stride;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                w[i][j] = (p0 + i < np && j < ncols) ? load(src[i] + j * col_stride) : kFull;
        }
        uint64_t t0 = 0;
        for (;;) {
            bool all = true;
#pragma unroll
            for (int i = 0; i < PB; ++i)
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (!(w[i][j] & kFull)) {
                        all = false;
                        w[i][j] = load(src[i] + j * col_stride);
                    }
            if (all)
                break;
            const uint64_t now = globaltimer_ns();
            if (!t0) {
                t0 = now;
            } else if (now - t0 > limit_ns) {
                ok = false;
                break;
            }
        }
#pragma unroll
        for (int i = 0; i < PB; ++i)
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (p0 + i < np) {
                    const float f = __uint_as_float((uint32_t)w[i][j]);
                    out[j] = (p0 + i == 0) ? f : out[j] + f;
                    if (j < ncols)  // clear the flag for the next launch
                        store(src[i] + j * col_stride, w[i][j] & 0xFFFFFFFFull);
                }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j)
        out[j] = (np == 0) ? __uint_as_float(own[j]) : out[j] + __uint_as_float(own[j]);
    return ok;
}

}  // namespace xch
}  // namespace dep
