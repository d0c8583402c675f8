// splitk_fma.cu -- weight-streaming warp split-K kernel on the FP32 FMA pipe.
//
// Computes y[B,N] = BF16(x[B,K] . W[N,K]^T) with FP32 accumulation for small
// batches (runtime.hybrid page, HybridAttention.__init__: warp split-K for up to
// 16 rows, the stock GEMM past that; runtime.dep page, module overview,
// precision paragraph: FP32 accumulation, BF16 outputs, split-K order of its own).
//
// Design (sm_103a):
//  * The weight is streamed exactly once.  Work units are (row tile t, k-tile kt)
//    pairs of TN weight rows x 256 columns, ordered row tile major; the grid's
//    persistent blocks take equal contiguous ranges of units (stream-K), so every
//    SM streams the same number of weight bytes whatever N and K are.
//  * One producer warp moves each unit's weight tile [TN x 256] and activation
//    tile [BC x 256] into a shared-memory ring with 2-D TMA bulk tensor copies
//    (completion on mbarriers; the weight with an L2 evict-first policy).
//  * Eight compute warps own R weight rows each.  Lane l owns columns 8l..8l+7
//    of every k-tile (one 16-byte shared load per row) and keeps one FP32 FMA
//    chain per (row, batch row); k-tiles are visited in increasing order.
//  * Where a block's range ends inside a row tile, the lanes' chains are summed
//    by an xor butterfly (16, 8, 4, 2, 1) and the warp's partials go to the
//    plan's workspace.  The last warp to arrive on the tile's counter (an integer
//    atomic) adds the partials in increasing block order, rounds to BF16 and
//    resets the counter.  No block waits for another and no float atomics are
//    used, so results are identical from run to run.
//  * Every wait is bounded in time; a warp that gives up records a code in the
//    device status word and leaves.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace dep {
namespace {

constexpr int kWarps = 8;                 // compute warps per block
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kKT = 256;                  // columns per k-tile: 32 lanes x 8
constexpr int kRowBytes = kKT * 2;        // one tile row in shared memory

// BC rows of x per pass, TN weight rows per tile (R = TN / 8 per compute warp).
template <int BC_, int TN_>
struct Shape {
    static constexpr int BC = BC_;
    static constexpr int TN = TN_;
    static constexpr int R = TN / kWarps;  // weight rows per compute warp
    static constexpr int STAGE_BYTES = (TN + BC) * kRowBytes;
    static_assert(R * BC <= 32, "one lane per (row, batch row) value in the epilogue");
};

__device__ __forceinline__ void unpack8(const uint4 v, float f[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);              // lower address: element 2i
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);  // element 2i + 1
    }
}

__device__ __forceinline__ uint16_t to_bf16(float v)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

template <int BC, int TN_>
__global__ void __launch_bounds__(kThreads, 1)
    splitk_fma_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                      uint16_t *__restrict__ y, int B, int N, int K, int stages,
                      float *__restrict__ ws, int *__restrict__ counters, int *__restrict__ status,
                      const Bounds bd, uint64_t limit_ns)
{
    constexpr int R = Shape<BC, TN_>::R, TN = TN_, STAGE_BYTES = Shape<BC, TN_>::STAGE_BYTES;
    extern __shared__ __align__(1024) uint8_t smem[];
    if (!dbg_ok((size_t)stages * STAGE_BYTES + 16 * (size_t)stages - 1, bd.smem, status))
        return;  // the ring and its barriers must lie in the launch's shared memory
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)stages * STAGE_BYTES);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + stages);

    const int64_t T = (N + TN - 1) / TN, KTILES = (K + kKT - 1) / kKT, U = T * KTILES;
    const int64_t C = gridDim.x, c = blockIdx.x;
    const int64_t u_begin = sk_begin(c, U, C), u_end = sk_begin(c + 1, U, C);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kWarps);
        }
        fence_mbar_init();
        griddep_launch_dependents();
    }
    __syncthreads();

    if (warp == kWarps) {  // ---------------- producer warp ----------------
        if (lane == 0) {
            prefetch_tmap(&tmW);
            prefetch_tmap(&tmX);
            const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
            // The weight is not written by preceding work: fill the ring with its
            // first tiles, then wait for the preceding grid before reading x.
            const SegOrder order(u_begin, u_end, KTILES);
            const int64_t pre = (u_end - u_begin) < stages ? (u_end - u_begin) : stages;
            UnitCursor cur(order);
            for (int64_t i = 0; i < pre; ++i, cur.next()) {
                const int64_t u = cur.u;
                mbar_arrive_expect_tx(full0 + 8 * (int)i, STAGE_BYTES);
                tma_load_2d(smem_u32(smem + (size_t)i * STAGE_BYTES), &tmW, (int)(u % KTILES) * kKT,
                            (int)(u / KTILES) * TN, full0 + 8 * (int)i, pol_w);
            }
            griddep_wait();
            UnitCursor cx(order);
            for (int64_t i = 0; i < pre; ++i, cx.next()) {
                const int64_t u = cx.u;
                tma_load_2d(smem_u32(smem + (size_t)i * STAGE_BYTES) + TN * kRowBytes, &tmX,
                            (int)(u % KTILES) * kKT, 0, full0 + 8 * (int)i, pol_x);
            }
            int s = (int)(pre % stages);
            uint32_t ph = pre == stages ? 1u : 0u;
            int64_t issued = pre;
            for (; !cur.done(); cur.next()) {
                const int64_t u = cur.u;
                if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, limit_ns)) {
                    record_status(status, DEP_DEV_TIMEOUT_PRODUCER);
                    break;
                }
                const uint32_t dst = smem_u32(smem + (size_t)s * STAGE_BYTES);
                mbar_arrive_expect_tx(full0 + 8 * s, STAGE_BYTES);
                const int t = (int)(u / KTILES), kt = (int)(u % KTILES);
                tma_load_2d(dst, &tmW, kt * kKT, t * TN, full0 + 8 * s, pol_w);
                tma_load_2d(dst + TN * kRowBytes, &tmX, kt * kKT, 0, full0 + 8 * s, pol_x);
                ++issued;
                if (++s == stages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            // Drain: the block must not exit while a copy into its shared memory
            // is in flight.  Walk back over the last `stages` fills.
            const int64_t n = issued < stages ? issued : stages;
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
        }
        return;
    }

    // ---------------- compute warps ----------------
    griddep_wait();  // workspace, counters and y may still be in use by the preceding grid
    float acc[R][BC];
    int s = 0;
    uint32_t ph = 0;
    const int64_t first_t = u_begin / KTILES;
    const SegOrder order(u_begin, u_end, KTILES);
    for (int64_t seg = 0; seg < order.m; ++seg) {
        const int64_t t = order.tile(seg);
        const int64_t seg_u0 = order.seg_begin(t), seg_end = order.seg_end(t);
        const bool whole = (seg_u0 == t * KTILES) && (seg_end == (t + 1) * KTILES);
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
            for (int b = 0; b < BC; ++b)
                acc[i][b] = 0.0f;

        for (int64_t u = seg_u0; u < seg_end; ++u) {
            if (!mbar_wait(full0 + 8 * s, ph, limit_ns)) {
                record_status(status, DEP_DEV_TIMEOUT_CONSUMER);
                return;
            }
            const uint8_t *st = smem + (size_t)s * STAGE_BYTES;
            float xv[BC][8];
#pragma unroll
            for (int b = 0; b < BC; ++b)
                unpack8(*reinterpret_cast<const uint4 *>(st + (TN + b) * kRowBytes + lane * 16), xv[b]);
#pragma unroll
            for (int i = 0; i < R; ++i) {
                float wv[8];
                unpack8(*reinterpret_cast<const uint4 *>(st + (warp * R + i) * kRowBytes + lane * 16), wv);
#pragma unroll
                for (int j = 0; j < 8; ++j)
#pragma unroll
                    for (int b = 0; b < BC; ++b)
                        acc[i][b] = __fmaf_rn(wv[j], xv[b][j], acc[i][b]);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(empty0 + 8 * s);
            if (++s == stages) {
                s = 0;
                ph ^= 1u;
            }
        }

        // ---- segment epilogue: warp sum, then direct store or split-K fix-up ----
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
            for (int b = 0; b < BC; ++b)
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1)
                    acc[i][b] += __shfl_xor_sync(0xFFFFFFFFu, acc[i][b], off);

        // lane L keeps value (i, b) = (L / BC, L % BC)
        float mine = 0.0f;
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
            for (int b = 0; b < BC; ++b)
                if (i * BC + b == lane)
                    mine = acc[i][b];
        const bool have = lane < R * BC;
        const int mb = lane % BC;
        const int row = warp * R + lane / BC;  // row within the tile
        const int64_t n = t * TN + row;

        if (whole) {
            if (have && mb < B && n < N && dbg_ok((int64_t)mb * N + n, bd.y, status))
                y[(int64_t)mb * N + n] = to_bf16(mine);
            continue;
        }
        const int slot = (t == first_t) ? 0 : 1;
        if (have && dbg_ok(((c * 2 + slot) * BC + mb) * TN + row, bd.ws, status))
            __stcg(&ws[((c * 2 + slot) * BC + mb) * TN + row], mine);
        __threadfence();
        __syncwarp();
        int prev = 0;
        if (lane == 0 && dbg_ok(t * kWarps + warp, bd.counters, status))
            prev = atomicAdd(&counters[t * kWarps + warp], 1);
        prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
        const int64_t c0 = sk_owner(t * KTILES, U, C), c1 = sk_owner(t * KTILES + KTILES - 1, U, C);
        if (prev != (int)(c1 - c0))
            continue;  // another block finishes this tile
        __threadfence();
        if (have) {
            // Sum the segments in increasing block order; up to 4 loads in flight.
            float sum = 0.0f;
            for (int64_t g0 = c0; g0 <= c1; g0 += 4) {
                float p[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int64_t cc = g0 + i;
                    const int sl = (t == sk_begin(cc, U, C) / KTILES) ? 0 : 1;
                    p[i] = cc <= c1 && dbg_ok(((cc * 2 + sl) * BC + mb) * TN + row, bd.ws, status)
                               ? __ldcg(&ws[((cc * 2 + sl) * BC + mb) * TN + row])
                               : 0.0f;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (g0 + i <= c1)
                        sum = (g0 + i == c0) ? p[i] : sum + p[i];
            }
            if (mb < B && n < N && dbg_ok((int64_t)mb * N + n, bd.y, status))
                y[(int64_t)mb * N + n] = to_bf16(sum);
        }
        if (lane == 0 && dbg_ok(t * kWarps + warp, bd.counters, status))
            counters[t * kWarps + warp] = 0;  // ready for the next launch
    }
}

// One block whose wait can never be satisfied: exercises the give-up path.
__global__ void selftest_timeout_kernel(int *status, uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (!mbar_wait(smem_u32(&bar), 0, limit_ns) && threadIdx.x == 0)
        record_status(status, DEP_DEV_TIMEOUT_CONSUMER);
}

template <class S>
size_t smem_bytes(int stages)
{
    return (size_t)stages * S::STAGE_BYTES + 2 * (size_t)stages * sizeof(uint64_t);
}

constexpr size_t kMaxSmem = kMaxDynamicSmem;

template <class S>
cudaError_t prepare()
{
    static std::atomic<uint64_t> devices{0};
    return set_smem_attr(splitk_fma_kernel<S::BC, S::TN>, devices);
}

// Call f with the Shape of (cols, tile rows); false if this build has no such kernel.
template <typename F>
bool with_shape(int cols, int tile_n, F &&f)
{
    switch (cols * 1000 + tile_n) {
    case 1032: f(Shape<1, 32>{}); return true;
    case 1064: f(Shape<1, 64>{}); return true;
    case 2032: f(Shape<2, 32>{}); return true;
    case 2064: f(Shape<2, 64>{}); return true;
    case 4032: f(Shape<4, 32>{}); return true;
    case 4064: f(Shape<4, 64>{}); return true;
    case 8032: f(Shape<8, 32>{}); return true;
    default: return false;
    }
}

template <class S>
cudaError_t run_shape(const dep_tactic_t &t, const RunArgs &a)
{
    constexpr int BC = S::BC, TN = S::TN;
    cudaError_t e = prepare<S>();
    if (e != cudaSuccess)
        return e;
    CUtensorMap tmW, tmX;
    if (encode_bf16_2d(&tmW, a.W, (uint64_t)a.K, (uint64_t)a.N, kKT, TN,
                       CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int64_t T = (a.N + TN - 1) / TN, KT = (a.K + kKT - 1) / kKT, U = T * KT;
    const int grid = (int)(U < t.ctas ? U : t.ctas);
    const size_t smem = smem_bytes<S>(t.stages);
    for (int32_t r0 = 0; r0 < a.B; r0 += BC) {
        const int32_t rows = a.B - r0 < BC ? a.B - r0 : BC;
        if (encode_bf16_2d(&tmX, a.x + (size_t)r0 * a.K, (uint64_t)a.K, (uint64_t)rows, kKT, BC,
                           CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        e = launch(splitk_fma_kernel<BC, TN>, dim3(grid), dim3(kThreads), smem, a.stream, a.pdl, tmW, tmX,
                   a.y + (size_t)r0 * a.N, rows, (int)a.N, (int)a.K, t.stages, a.ws, a.counters, a.status,
                   a.bounds(rows, smem), a.wait_limit_ns);
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

// Default tile height for a column count: 32 rows (one 16-byte load per lane
// per row; smaller boxes bring the first data in sooner).
int tile_rows(int cols)
{
    return (cols == 1 || cols == 2 || cols == 4 || cols == 8) ? 32 : 0;
}

}  // namespace

bool fma_valid(const dep_tactic_t &t)
{
    if (t.kind != DEP_KIND_SPLITK_FMA || t.ctas < 1 || t.tile_k != kKT)
        return false;
    if (t.stages < 2 || t.stages > 16)
        return false;
    size_t smem = 0;
    if (!with_shape(t.cols, t.tile_n, [&](auto sh) { smem = smem_bytes<decltype(sh)>(t.stages); }))
        return false;
    return smem <= kMaxSmem;
}

int64_t fma_units(const dep_tactic_t &t, int64_t N, int64_t K)
{
    return ((N + t.tile_n - 1) / t.tile_n) * ((K + kKT - 1) / kKT);
}

size_t fma_ws_per_cta(const dep_tactic_t &t)
{
    return 2 * (size_t)t.cols * (size_t)t.tile_n;  // head and tail segment partials
}

size_t fma_counters(const dep_tactic_t &t, int64_t N)
{
    return (size_t)((N + t.tile_n - 1) / t.tile_n) * kWarps;
}

int fma_blocks_per_sm(const dep_tactic_t &t)
{
    int n = 0;
    with_shape(t.cols, t.tile_n, [&](auto sh) {
        using S = decltype(sh);
        if (prepare<S>() != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, splitk_fma_kernel<S::BC, S::TN>, kThreads,
                                                          smem_bytes<S>(t.stages)) != cudaSuccess)
            n = 0;
    });
    return n;
}

cudaError_t fma_prepare_device()
{
    cudaError_t e = cudaSuccess;
    for (int cols : {1, 2, 4, 8})
        for (int tn : {32, 64})
            with_shape(cols, tn, [&](auto sh) {
                const cudaError_t r = prepare<decltype(sh)>();
                if (r != cudaSuccess)
                    e = r;
            });
    return e;
}

cudaError_t fma_run(const dep_tactic_t &t, const RunArgs &a)
{
    cudaError_t e = cudaErrorInvalidValue;
    with_shape(t.cols, t.tile_n, [&](auto sh) { e = run_shape<decltype(sh)>(t, a); });
    return e;
}

cudaError_t selftest_timeout(int32_t limit_us, int32_t *code)
{
    int *d = nullptr;
    cudaError_t e = cudaMalloc(&d, sizeof(int));
    if (e != cudaSuccess)
        return e;
    e = cudaMemset(d, 0, sizeof(int));
    if (e == cudaSuccess) {
        selftest_timeout_kernel<<<1, 32>>>(d, (uint64_t)limit_us * 1000ull);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess)
        e = cudaDeviceSynchronize();
    int h = 0;
    if (e == cudaSuccess)
        e = cudaMemcpy(&h, d, sizeof(int), cudaMemcpyDeviceToHost);
    cudaFree(d);
    *code = h;
    return e;
}

}  // namespace dep

// ---------------------------------------------------------------------------
// dep_projection_run_static: the split-K FMA kernel with its scratch in a fixed
// array compiled into this library, for callers that must not allocate.
//
// Who cannot allocate: code that runs inside a device-memory allocator or pool
// (allocating there would re-enter the allocator), hosts that reserve all device
// memory up front and forbid any other allocation, and latency-critical paths
// where cudaMalloc's implicit synchronisation is not acceptable.  Such callers
// cannot build a plan, because a plan allocates its workspace.
//
// The scratch (status word, tile counters, split-K partials) lives in one
// file-scope __device__ array of kStaticScratchBytes.  Every GPU that loads this
// library holds it until the process exits.  Host code cannot use the array's
// name as a device address (it is a host-side stand-in), so the first call on a
// device looks the address up with cudaGetSymbolAddress while that device is
// current and keeps it; that first call should therefore come before any stream
// capture.  All calls share the array and it keeps the last call's contents:
// each call clears the counters and the status word (they must start at zero)
// on its stream; the partials are always written before they are read.  Calls
// that overlap on the GPU race on the array.
// ---------------------------------------------------------------------------
#include <mutex>

namespace dep {
namespace {

constexpr size_t kStaticScratchBytes = 1u << 20;        // 1 MiB in total
constexpr size_t kStaticStatusBytes = 256;              // status word (padded)
constexpr size_t kStaticCounterBytes = 256u * 1024u;    // 65536 tile counters
constexpr size_t kStaticPartialBytes = kStaticScratchBytes - kStaticStatusBytes - kStaticCounterBytes;
constexpr int kStaticMaxDevices = 64;
constexpr int64_t kStaticMaxRows = 262144;  // weight rows: 32-row tiles x 8 counters fit the counter area

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

struct StaticDevice {
    bool ready;
    unsigned char *scratch;  // device address of g_static_scratch on this device
    int sm_count;
};
std::mutex g_static_mutex;
StaticDevice g_static_devices[kStaticMaxDevices];

// Once per device, with that device current.
cudaError_t static_device(int dev, StaticDevice *out)
{
    std::lock_guard<std::mutex> lock(g_static_mutex);
    StaticDevice &d = g_static_devices[dev];
    if (!d.ready) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess)
            return e;
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return e;
        d.scratch = static_cast<unsigned char *>(p);
        d.sm_count = sms;
        d.ready = true;
    }
    *out = d;
    return cudaSuccess;
}

}  // namespace
}  // namespace dep

extern "C" dep_status_t dep_projection_run_static(const void *x, const void *W, void *y, int64_t N,
                                                  int64_t K, int32_t B, void *stream)
{
    using namespace dep;
    if (B < 0 || N < 1 || K < 8)
        return DEP_ERR_INVALID_ARG;
    if (K % 8)
        return DEP_ERR_MISALIGNED;
    if (N > kStaticMaxRows || K > INT32_MAX)
        return DEP_ERR_UNSUPPORTED;  // beyond the fixed scratch array's stated limit
    if (B == 0)
        return DEP_OK;
    if (!x || !W || !y)
        return DEP_ERR_INVALID_ARG;
    const uintptr_t px = reinterpret_cast<uintptr_t>(x), pw = reinterpret_cast<uintptr_t>(W),
                    py = reinterpret_cast<uintptr_t>(y);
    if ((px | pw | py) & 15u)
        return DEP_ERR_MISALIGNED;
    const size_t xb = (size_t)B * K * 2, wb = (size_t)N * K * 2, yb = (size_t)B * N * 2;
    if ((py < px + xb && px < py + yb) || (py < pw + wb && pw < py + yb))
        return DEP_ERR_INVALID_ARG;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kStaticMaxDevices) {
        cudaGetLastError();
        return DEP_ERR_CUDA;
    }
    StaticDevice sd;
    if (static_device(dev, &sd) != cudaSuccess) {
        cudaGetLastError();
        return DEP_ERR_CUDA;
    }

    dep_tactic_t t{};
    t.max_rows = B;
    t.kind = DEP_KIND_SPLITK_FMA;
    t.cols = B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : 8;
    t.tile_n = tile_rows(t.cols);
    t.tile_k = kKT;
    t.stages = t.cols >= 8 ? 6 : 4;
    t.ctas = sd.sm_count;
    const int64_t U = fma_units(t, N, K);
    const int64_t grid = U < t.ctas ? U : t.ctas;
    const size_t counters = fma_counters(t, N);
    if (counters * sizeof(int) > kStaticCounterBytes ||
        (size_t)grid * fma_ws_per_cta(t) * sizeof(float) > kStaticPartialBytes)
        return DEP_ERR_UNSUPPORTED;  // larger than the fixed scratch array

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(sd.scratch, 0, kStaticStatusBytes + counters * sizeof(int), s) != cudaSuccess) {
        cudaGetLastError();
        return DEP_ERR_CUDA;
    }
    RunArgs a;
    a.x = static_cast<const uint16_t *>(x);
    a.W = static_cast<const uint16_t *>(W);
    a.y = static_cast<uint16_t *>(y);
    a.B = B;
    a.N = N;
    a.K = K;
    a.status = reinterpret_cast<int *>(sd.scratch);
    a.counters = reinterpret_cast<int *>(sd.scratch + kStaticStatusBytes);
    a.n_counters = kStaticCounterBytes / sizeof(int);
    a.ws = reinterpret_cast<float *>(sd.scratch + kStaticStatusBytes + kStaticCounterBytes);
    a.ws_floats = kStaticPartialBytes / sizeof(float);
    a.stream = s;
    a.wait_limit_ns = 1000000000ull;
    if (fma_run(t, a) != cudaSuccess) {
        cudaGetLastError();
        return DEP_ERR_CUDA;
    }
    return DEP_OK;
}
