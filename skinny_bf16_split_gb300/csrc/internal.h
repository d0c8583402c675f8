// internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "../../include/dep_projection.h"

namespace dep {

// Sizes of what one launch may index, for the bounds checks of the DEP_DEBUG
// build (elements of y, of the split-K partials, counters and exchange words,
// and bytes of dynamic shared memory).  Passed to every kernel; other builds
// compile the checks away.
struct Bounds {
    unsigned long long y, ws, counters, xch, smem;
};

// One launch's operands and the plan-owned scratch it may use.
struct RunArgs {
    const uint16_t *x;  // [B, K] BF16 bits, device
    const uint16_t *W;  // [N, K]
    uint16_t *y;        // [B, N]
    int32_t B;
    int64_t N, K;
    float *ws;          // split-K partials
    size_t ws_floats;
    int *counters;      // per-tile arrival counters (zero between launches)
    size_t n_counters;
    unsigned long long *xch = nullptr;  // K-piece exchange words (flags clear between launches)
    size_t xch_words = 0;
    int *status;        // device status word (0 = fine)
    cudaStream_t stream;
    uint64_t wait_limit_ns;
    // Programmatic dependent launch: the kernel may start while the preceding
    // grid in the stream finishes; it streams its first weight stages before
    // waiting for that grid (the weight must not be written by preceding work).
    bool pdl = false;
    // The wide kernel also stores the partials its blocks reduce themselves.
    bool keep_pieces = false;
    // What a launch of `y_rows` batch rows with `smem` bytes of shared memory may index.
    Bounds bounds(int64_t y_rows, size_t smem) const
    {
        return Bounds{(unsigned long long)y_rows * (unsigned long long)N, ws_floats, n_counters, xch_words, smem};
    }
};

// Shared memory a block of any kernel here may use (the sm_100-family opt-in maximum).
constexpr int kMaxDynamicSmem = 227 * 1024;

// Raise a kernel's dynamic shared-memory limit on the current device, once per
// device (the attribute belongs to the device's context).  `devices` is the
// kernel's own record of the devices already done (one bit per device < 64).
template <typename Kernel>
cudaError_t set_smem_attr(Kernel kernel, std::atomic<uint64_t> &devices)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0;
    if (bit && (devices.load(std::memory_order_acquire) & bit))
        return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynamicSmem);
    // All of the unified L1 as shared memory: no kernel here reads through L1,
    // and a block of the next grid in the stream (programmatic dependent launch)
    // can then sit beside a running block whenever the two rings fit together.
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess && bit)
        devices.fetch_or(bit, std::memory_order_release);
    return e;
}

// Set the attribute of every kernel instantiation on the current device
// (called when a plan is made, so that no first launch happens inside a
// stream capture).
cudaError_t fma_prepare_device();
cudaError_t tc_prepare_device();
cudaError_t rows_prepare_device();
cudaError_t tcs_prepare_device();
cudaError_t wide_prepare_device();
cudaError_t cluster_prepare_device();
cudaError_t xm_prepare_device();
cudaError_t mma_rows_prepare_device();

// Launch with the programmatic-stream-serialisation attribute when `pdl` is set.
template <typename Kernel, typename... Args>
cudaError_t launch(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                   Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Stream-K split: U work units over C blocks, block c owns [begin(c), begin(c+1)).
__host__ __device__ inline int64_t sk_begin(int64_t c, int64_t U, int64_t C)
{
    return (c * U) / C;
}
// The block owning unit u (the c with begin(c) <= u < begin(c+1); needs U >= C).
__host__ __device__ inline int64_t sk_owner(int64_t u, int64_t U, int64_t C)
{
    return ((u + 1) * C - 1) / U;
}

// Order in which a block visits its units: the segment of its last tile first,
// then the segment of its first tile, then the whole tiles in between.  Both
// split tiles a block shares with its neighbours are thus finished (and their
// split-K fix-up done) early, and the block ends on a whole tile whenever its
// range holds one.  Units inside a segment keep increasing k order, so the
// arithmetic of every output does not depend on this order.
struct SegOrder {
    int64_t u_begin, u_end, ktiles, t_first, t_last, m;
    __host__ __device__ SegOrder(int64_t ub, int64_t ue, int64_t kt)
        : u_begin(ub), u_end(ue), ktiles(kt), t_first(ub / kt), t_last(ue > ub ? (ue - 1) / kt : ub / kt),
          m(ue > ub ? t_last - t_first + 1 : 0)
    {
    }
    __host__ __device__ int64_t tile(int64_t i) const
    {
        return m >= 2 ? (i == 0 ? t_last : t_first + i - 1) : t_first;
    }
    __host__ __device__ int64_t seg_begin(int64_t t) const
    {
        return u_begin > t * ktiles ? u_begin : t * ktiles;
    }
    __host__ __device__ int64_t seg_end(int64_t t) const
    {
        return u_end < (t + 1) * ktiles ? u_end : (t + 1) * ktiles;
    }
};

// Walks a block's units in SegOrder.
struct UnitCursor {
    SegOrder o;
    int64_t i, u, end;
    __host__ __device__ explicit UnitCursor(const SegOrder &order) : o(order), i(0), u(0), end(0)
    {
        if (o.m > 0) {
            u = o.seg_begin(o.tile(0));
            end = o.seg_end(o.tile(0));
        }
    }
    __host__ __device__ bool done() const { return i >= o.m; }
    __host__ __device__ void next()
    {
        if (++u < end)
            return;
        if (++i < o.m) {
            u = o.seg_begin(o.tile(i));
            end = o.seg_end(o.tile(i));
        }
    }
};

// ---- split-K FMA tactic (splitk_fma.cu) ----
bool fma_valid(const dep_tactic_t &t);
int64_t fma_units(const dep_tactic_t &t, int64_t N, int64_t K);  // stream-K work units
size_t fma_ws_per_cta(const dep_tactic_t &t);                     // partial floats per block
size_t fma_counters(const dep_tactic_t &t, int64_t N);
int fma_blocks_per_sm(const dep_tactic_t &t);  // occupancy, 0 if it cannot launch
cudaError_t fma_run(const dep_tactic_t &t, const RunArgs &a);
cudaError_t selftest_timeout(int32_t limit_us, int32_t *code);

// ---- tcgen05 tactic (tc_gemm.cu) ----
bool tc_valid(const dep_tactic_t &t);
int64_t tc_units(const dep_tactic_t &t, int64_t N, int64_t K);
size_t tc_xch_words_per_cta(const dep_tactic_t &t);              // exchange words per block
size_t tc_xch_words(const dep_tactic_t &t, int64_t N, int64_t K);  // exchange words of a launch
int tc_blocks_per_sm(const dep_tactic_t &t);
cudaError_t tc_run(const dep_tactic_t &t, const RunArgs &a);

// ---- tcgen05 tactic with fixed K pieces, dynamically scheduled (tc_split.cu) ----
bool tcs_valid(const dep_tactic_t &t);
size_t tcs_xch_words(const dep_tactic_t &t, int64_t N, int64_t K);  // every piece's exchange word
size_t tcs_counters(const dep_tactic_t &t, int64_t N);               // the last 2 counters
int tcs_blocks_per_sm(const dep_tactic_t &t);
int64_t tcs_items(const dep_tactic_t &t, int64_t N, int64_t K);      // (tile, piece) items of a launch
cudaError_t tcs_run(const dep_tactic_t &t, const RunArgs &a);       // uses the last 2 counters
cudaError_t tcs_selftest_exchange(unsigned long long *xch, size_t xch_words, int *counters, int *status,
                                  uint64_t limit_ns, cudaStream_t stream);

// ---- tcgen05 tactic for wide batches, groups of tiles per x slice (tc_wide.cu) ----
bool wide_valid(const dep_tactic_t &t);
int64_t wide_units(const dep_tactic_t &t, int64_t N, int64_t K);  // stream-K work units
size_t wide_ws_per_cta(const dep_tactic_t &t);                    // partial floats per block (two slots)
size_t wide_flags_per_cta(const dep_tactic_t &t);                 // flag ints per block (the first counters)
int wide_blocks_per_sm(const dep_tactic_t &t);
cudaError_t wide_run(const dep_tactic_t &t, const RunArgs &a);

// ---- tcgen05 tactic for wide batches, a cluster of CTAs per group (tc_cluster.cu) ----
bool cluster_valid(const dep_tactic_t &t);
cudaError_t cluster_run(const dep_tactic_t &t, const RunArgs &a);

// ---- tcgen05 tactic for wide batches, x on the MMA's M side (tc_xm.cu) ----
bool xm_valid(const dep_tactic_t &t);
int64_t xm_tiles(const dep_tactic_t &t, int64_t N);
// Deepest ring (2..16 stages, 0 if none) of tiles of tile_n weight rows, stages
// of tile_k columns and cols = 128 or 256 batch rows per pass, when the pass's
// x blocks have mr = 64 or 128 rows.
int xm_stages_fit(int32_t tile_n, int32_t tile_k, int32_t cols, int mr);
cudaError_t xm_run(const dep_tactic_t &t, const RunArgs &a);

// ---- warp-level MMA tactic for small weights (mma_rows.cu) ----
bool mma_rows_valid(const dep_tactic_t &t);
int64_t mma_rows_tiles(const dep_tactic_t &t, int64_t N);
cudaError_t mma_rows_run(const dep_tactic_t &t, const RunArgs &a);

// ---- whole-row tactic (rows_gemv.cu) ----
bool rows_valid(const dep_tactic_t &t);
bool rows_fits(const dep_tactic_t &t, int64_t K);  // x and the ring fit in shared memory
int64_t rows_tiles(const dep_tactic_t &t, int64_t N);
int rows_blocks_per_sm(const dep_tactic_t &t, int64_t K);
cudaError_t rows_run(const dep_tactic_t &t, const RunArgs &a);  // uses the last 2 counters

// ---- zero-copy staging for the host-buffer entry point (staging.cu) ----
// Copy n BF16 elements src -> dst (16-byte aligned; either side may be mapped
// host memory).  after_preceding: launched with programmatic dependent launch,
// waits for the preceding grid before reading src.
cudaError_t stage_copy(const uint16_t *src, uint16_t *dst, size_t n, bool after_preceding, cudaStream_t stream);

// ---- TMA descriptors (tma.cpp) ----
// 2-D BF16 tensor map over a row-major [outer, inner] array with a row pitch of
// `inner` elements; box = [box_outer rows, box_inner elements]; out-of-range
// elements read as zero.
CUresult encode_bf16_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer,
                        uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);
// The same matrix as {64, outer, inner / 64} column blocks (inner % 64 == 0):
// one box {64, box_rows, blocks} equals `blocks` 2-D boxes {64, box_rows} with
// the 128-byte swizzle, side by side in shared memory.
CUresult encode_bf16_3d_blocks(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer,
                               uint32_t box_rows, uint32_t blocks);

}  // namespace dep
