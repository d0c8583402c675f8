// rows_gemv.cu -- warp split-K over whole weight rows, dynamically scheduled.
//
// Computes y[B,N] = BF16(x[B,K] . W[N,K]^T) with FP32 accumulation for the
// smallest batches (runtime.hybrid page, HybridAttention.__init__: warp split-K
// for the few-row batches; runtime.dep page, module overview, precision
// paragraph: FP32 accumulation, BF16 outputs).
//
// Design (sm_103a):
//  * Work items are tiles of TN = 8 * RW whole weight rows (all of K).  Each
//    output is summed by exactly one warp -- K split across its 32 lanes, lane
//    chains reduced by an xor butterfly -- so no partial sums cross blocks and
//    there is no split-K fix-up at all.  The result is independent of the
//    schedule and equals the stream-K FMA tactic's order for a tile that one
//    block owns whole: lane l takes columns 256 kt + 8 l + j, kt then j
//    increasing, with +0 past column K-1.
//  * Blocks take tiles dynamically: tile blockIdx.x first, then the next free
//    tile from an integer counter, so a block that streams faster takes more
//    tiles and all blocks finish together.  The last block to finish resets the
//    counters for the next launch.
//  * x [BC x K] is loaded once per block into shared memory (bulk copies) and
//    stays there; the weight streams through a ring of stages of TN rows x KC
//    columns, each stage KC / 256 2-D TMA boxes of TN rows x 256 columns (a
//    stage is laid out box after box); rows past N-1 and columns past K-1 read
//    as zero.  (Per-row 1-D bulk copies of the same stages measured 30-60 %
//    slower on GB300.)
//  * Every wait is bounded in time; a warp that gives up records a code in the
//    device status word and leaves after the block's copies have landed.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace dep {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kSub = 256;  // columns per lane sweep: 32 lanes x 8
constexpr size_t kMaxSmem = kMaxDynamicSmem;

// 1-D bulk copy global -> shared, completion on an mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void unpack8(const uint4 v, float f[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// Shared-memory layout: [x: BC rows x K_pad bf16][ring: stages x (KC/256 boxes of TN x 256) bf16]
//                       [barriers: full[stages], empty[stages], xbar][tags[stages]]
struct RowsLayout {
    size_t x_bytes, stage_bytes, ring, bars, tags, total;
    __host__ __device__ RowsLayout(int BC, int TN, int KC, int stages, int64_t K)
    {
        const int64_t kpad = ((K + kSub - 1) / kSub) * kSub;
        x_bytes = (size_t)BC * kpad * 2;
        stage_bytes = (size_t)TN * KC * 2;
        ring = x_bytes;  // x_bytes is a multiple of 512
        bars = ring + (size_t)stages * stage_bytes;
        tags = bars + (2 * (size_t)stages + 1) * 8;
        total = tags + (size_t)stages * 8;
    }
};

template <int BC, int RW>
__global__ void __launch_bounds__(kThreads, 1)
    rows_gemv_kernel(const uint16_t *__restrict__ x, const __grid_constant__ CUtensorMap tmW, uint16_t *__restrict__ y,
                     int B, int N, int K, int KC, int stages, int *__restrict__ counters,
                     int *__restrict__ status, const Bounds bd, uint64_t limit_ns)
{
    constexpr int TN = kWarps * RW;
    extern __shared__ __align__(1024) uint8_t smem[];
    const RowsLayout L(BC, TN, KC, stages, K);
    if (!dbg_ok(L.total - 1, bd.smem, status))
        return;  // x, the ring and the barriers must lie in the launch's shared memory
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    int2 *tags = reinterpret_cast<int2 *>(smem + L.tags);  // (tile, chunk) per stage; tile < 0: end
    const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * stages, xbar = empty0 + 8 * stages;
    const int T = (N + TN - 1) / TN, NCH = (K + KC - 1) / KC;
    const int64_t kpad = ((int64_t)(K + kSub - 1) / kSub) * kSub;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int *grab = counters, *done = counters + 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kWarps);
        }
        mbar_init(xbar, 1);
        fence_mbar_init();
        griddep_launch_dependents();
    }
    __syncthreads();

    if (warp == kWarps) {  // ---------------- producer warp ----------------
        if (lane == 0) {
            prefetch_tmap(&tmW);
            const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
            // One stage: `chunk` of tile `tile` (TN rows x up to KC columns).
            auto issue = [&](int tile, int chunk, int st) {
                const int k0 = chunk * KC, cols = K - k0 < KC ? K - k0 : KC;
                const int row0 = tile * TN;
                tags[st] = make_int2(tile, chunk);
                const int nsub = (cols + kSub - 1) / kSub;
                mbar_arrive_expect_tx(full0 + 8 * st, (uint32_t)(nsub * TN * kSub * 2));
                const uint32_t dst = smem_u32(smem + L.ring + (size_t)st * L.stage_bytes);
                for (int q = 0; q < nsub; ++q)
                    tma_load_2d(dst + (uint32_t)(q * TN * kSub * 2), &tmW, k0 + q * kSub, row0, full0 + 8 * st,
                                pol_w);
            };
            // Phase 1: the weight is not written by preceding work -- fill the ring
            // with the first chunks of this block's first tile (tile blockIdx.x).
            int tile = blockIdx.x;
            const int pre = NCH < stages ? NCH : stages;
            for (int i = 0; i < pre; ++i)
                issue(tile, i, i);
            int s = pre % stages, chunk = pre;
            uint32_t ph = pre == stages ? 1u : 0u;
            int64_t issued = pre;
            // Phase 2: after the preceding grid -- x, then tiles taken from the counter.
            griddep_wait();
            mbar_arrive_expect_tx(xbar, (uint32_t)(B * K * 2));
            for (int b = 0; b < B; ++b)
                bulk_load(smem_u32(xs + (size_t)b * kpad), x + (size_t)b * K, (uint32_t)K * 2, xbar, pol_x);
            if (chunk == NCH) {
                chunk = 0;
                tile = (int)gridDim.x + atomicAdd(grab, 1);
            }
            bool ok = true;
            for (;;) {
                if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, limit_ns)) {
                    record_status(status, DEP_DEV_TIMEOUT_PRODUCER);
                    ok = false;
                    break;
                }
                if (tile >= T) {  // end of the stream: an empty stage tagged -1
                    tags[s] = make_int2(-1, 0);
                    mbar_arrive(full0 + 8 * s);
                    break;
                }
                issue(tile, chunk, s);
                ++issued;
                if (++s == stages) {
                    s = 0;
                    ph ^= 1u;
                }
                if (++chunk == NCH) {
                    chunk = 0;
                    tile = (int)gridDim.x + atomicAdd(grab, 1);
                }
            }
            // Drain: every copy into this block's shared memory has landed.
            if (!mbar_wait(xbar, 0, limit_ns))
                record_status(status, DEP_DEV_TIMEOUT_PRODUCER);
            // Walk back over the most recent fills from stage s.  After an end
            // marker, stage s holds the marker, so at most stages - 1 copies can
            // still be in flight; after a give-up, stage s was never refilled.
            const int64_t cap = ok ? stages - 1 : stages;
            const int64_t n = issued < cap ? issued : cap;
            int ds = s;
            uint32_t dph = ph;
            for (int64_t i = 0; i < n; ++i) {
                if (--ds < 0) {
                    ds = stages - 1;
                    dph ^= 1u;
                }
                if (!mbar_wait(full0 + 8 * ds, dph, limit_ns))
                    record_status(status, DEP_DEV_TIMEOUT_PRODUCER);
            }
            // The last block to finish taking tiles resets the counters.
            if (atomicAdd(done, 1) == (int)gridDim.x - 1) {
                *grab = 0;
                *done = 0;
            }
        }
        return;
    }

    // ---------------- compute warps ----------------
    // x rows past B read as zero (their outputs are not stored).
    for (int64_t i = threadIdx.x; i < (int64_t)(BC - B) * kpad; i += kWarps * 32)
        xs[(size_t)B * kpad + i] = 0;
    for (int64_t i = threadIdx.x; i < (int64_t)B * (kpad - K); i += kWarps * 32) {
        const int64_t b = i / (kpad - K), k = K + i % (kpad - K);
        xs[b * kpad + k] = 0;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");  // compute warps only
    if (!mbar_wait(xbar, 0, limit_ns)) {
        record_status(status, DEP_DEV_TIMEOUT_CONSUMER);
        return;
    }
    griddep_wait();  // y may still be in use by the preceding grid
    const int KTILES = (K + kSub - 1) / kSub;
    float acc[RW][BC];
    int s = 0;
    uint32_t ph = 0;
    for (;;) {
        if (!mbar_wait(full0 + 8 * s, ph, limit_ns)) {
            record_status(status, DEP_DEV_TIMEOUT_CONSUMER);
            return;
        }
        const int2 tag = tags[s];
        if (tag.x < 0)
            break;
        const int tile = tag.x, chunk = tag.y;
        if (chunk == 0) {
#pragma unroll
            for (int i = 0; i < RW; ++i)
#pragma unroll
                for (int b = 0; b < BC; ++b)
                    acc[i][b] = 0.0f;
        }
        const uint8_t *st = smem + L.ring + (size_t)s * L.stage_bytes;
        const int kt0 = chunk * (KC / kSub);
        const int nkt = (KTILES - kt0) < KC / kSub ? (KTILES - kt0) : KC / kSub;
        const int row0 = tile * TN;
        for (int q = 0; q < nkt; ++q) {
            const int64_t k = (int64_t)(kt0 + q) * kSub + lane * 8;
            float xv[BC][8];
#pragma unroll
            for (int b = 0; b < BC; ++b)
                unpack8(*reinterpret_cast<const uint4 *>(xs + (size_t)b * kpad + k), xv[b]);
#pragma unroll
            for (int i = 0; i < RW; ++i) {
                const int r = warp * RW + i;
                float wv[8];
                // past column K-1 or row N-1 the box read zeros (and x is zero past K-1)
                unpack8(*reinterpret_cast<const uint4 *>(st + ((size_t)(q * TN + r) * kSub + lane * 8) * 2), wv);
#pragma unroll
                for (int j = 0; j < 8; ++j)
#pragma unroll
                    for (int b = 0; b < BC; ++b)
                        acc[i][b] = __fmaf_rn(wv[j], xv[b][j], acc[i][b]);
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(empty0 + 8 * s);
        if (++s == stages) {
            s = 0;
            ph ^= 1u;
        }
        if (chunk != NCH - 1)
            continue;
        // ---- tile done: warp sum and store ----
#pragma unroll
        for (int i = 0; i < RW; ++i)
#pragma unroll
            for (int b = 0; b < BC; ++b)
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1)
                    acc[i][b] += __shfl_xor_sync(0xFFFFFFFFu, acc[i][b], off);
#pragma unroll
        for (int i = 0; i < RW; ++i)
#pragma unroll
            for (int b = 0; b < BC; ++b)
                if (lane == i * BC + b) {
                    const int64_t n = (int64_t)row0 + warp * RW + i;
                    if (b < B && n < N && dbg_ok((int64_t)b * N + n, bd.y, status))
                        y[(int64_t)b * N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[i][b]));
                }
    }
}

template <int BC, int RW>
cudaError_t prepare()
{
    static std::atomic<uint64_t> devices{0};
    return set_smem_attr(rows_gemv_kernel<BC, RW>, devices);
}

template <typename F>
bool with_rows_shape(int cols, int tile_n, F &&f)
{
    switch (cols * 1000 + tile_n) {
    case 1008: f(std::integral_constant<int, 1>{}, std::integral_constant<int, 1>{}); return true;
    case 1016: f(std::integral_constant<int, 1>{}, std::integral_constant<int, 2>{}); return true;
    case 2008: f(std::integral_constant<int, 2>{}, std::integral_constant<int, 1>{}); return true;
    case 2016: f(std::integral_constant<int, 2>{}, std::integral_constant<int, 2>{}); return true;
    case 4008: f(std::integral_constant<int, 4>{}, std::integral_constant<int, 1>{}); return true;
    case 4016: f(std::integral_constant<int, 4>{}, std::integral_constant<int, 2>{}); return true;
    default: return false;
    }
}

}  // namespace

bool rows_valid(const dep_tactic_t &t)
{
    if (t.kind != DEP_KIND_ROWS || t.ctas < 1 || t.stages < 2 || t.stages > 16)
        return false;
    if (t.tile_k != 1024 && t.tile_k != 2048 && t.tile_k != 4096)
        return false;
    bool known = false;
    with_rows_shape(t.cols, t.tile_n, [&](auto, auto) { known = true; });
    return known;
}

bool rows_fits(const dep_tactic_t &t, int64_t K)
{
    return RowsLayout(t.cols, t.tile_n, t.tile_k, t.stages, K).total <= kMaxSmem;
}

int64_t rows_tiles(const dep_tactic_t &t, int64_t N)
{
    return (N + t.tile_n - 1) / t.tile_n;
}

int rows_blocks_per_sm(const dep_tactic_t &t, int64_t K)
{
    int n = 0;
    with_rows_shape(t.cols, t.tile_n, [&](auto bc, auto rw) {
        constexpr int BC = decltype(bc)::value, RW = decltype(rw)::value;
        if (prepare<BC, RW>() != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &n, rows_gemv_kernel<BC, RW>, kThreads,
                RowsLayout(BC, 8 * RW, t.tile_k, t.stages, K).total) != cudaSuccess)
            n = 0;
    });
    return n;
}

cudaError_t rows_prepare_device()
{
    cudaError_t e = cudaSuccess;
    for (int cols : {1, 2, 4})
        for (int tn : {8, 16})
            with_rows_shape(cols, tn, [&](auto bc, auto rw) {
                const cudaError_t r = prepare<decltype(bc)::value, decltype(rw)::value>();
                if (r != cudaSuccess)
                    e = r;
            });
    return e;
}

cudaError_t rows_run(const dep_tactic_t &t, const RunArgs &a)
{
    cudaError_t e = cudaErrorInvalidValue;
    with_rows_shape(t.cols, t.tile_n, [&](auto bc, auto rw) {
        constexpr int BC = decltype(bc)::value, RW = decltype(rw)::value;
        e = prepare<BC, RW>();
        if (e != cudaSuccess)
            return;
        const int64_t T = (a.N + 8 * RW - 1) / (8 * RW);
        const int grid = (int)(T < t.ctas ? T : t.ctas);
        const size_t smem = RowsLayout(BC, 8 * RW, t.tile_k, t.stages, a.K).total;
        CUtensorMap tmW;
        if (encode_bf16_2d(&tmW, a.W, (uint64_t)a.K, (uint64_t)a.N, kSub, 8 * RW, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS) {
            e = cudaErrorInvalidValue;
            return;
        }
        for (int32_t r0 = 0; r0 < a.B && e == cudaSuccess; r0 += BC) {
            const int32_t rows = a.B - r0 < BC ? a.B - r0 : BC;
            e = launch(rows_gemv_kernel<BC, RW>, dim3(grid), dim3(kThreads), smem, a.stream, a.pdl,
                       a.x + (size_t)r0 * a.K, tmW, a.y + (size_t)r0 * a.N, rows, (int)a.N, (int)a.K,
                       t.tile_k, t.stages, a.counters + a.n_counters - 2, a.status, a.bounds(rows, smem),
                       a.wait_limit_ns);
        }
    });
    return e;
}

}  // namespace dep
