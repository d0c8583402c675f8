// tc_wide.cu -- tcgen05 tactic for wide batches: several weight tiles per x slice.
//
// Computes y[B,N] = BF16(x[B,K] . W[N,K]^T), BF16 products accumulated in FP32,
// for the batches past the split-K rows (runtime.hybrid page,
// HybridAttention.__init__: past them the projection runs the stock
// FP32-accumulated BF16 GEMM; runtime.dep page, DepProjection.run).
//
// Why another kernel: with one 128-row weight tile per x slice a block takes in
// NT x 128 B of x for every 16 KB of weight, three times the weight bytes at
// NT = 256, and what one SM can take in from L2 -- not HBM -- then bounds the
// call.  Here a block streams a group of G = 2 or 4 consecutive 128-row tiles
// against each x slice and issues one M = 128 MMA per tile with the same x
// descriptor, so the x bytes per weight byte fall by G.
//
// Design (sm_103a, one CTA per SM, no clusters, no multicast):
//  * Swap-AB as in the other tensor-core kernels: MMA M = 128 weight rows, N =
//    the batch padded to NT (32..256), K = 16 per instruction; D in TMEM.  A
//    group's accumulator is G x NT TMEM columns (tile g at column g NT); two
//    buffers where 2 G NT <= 512, else one (G = 2, NT = 256 fills TMEM).
//  * Work units are (group, tile_k-column k-tile) pairs; the persistent blocks
//    take equal contiguous ranges (stream-K).  A block visits its last group
//    first, then the whole groups in between, then its first group.
//  * Warp 0: TMA producer (per stage G weight boxes [128 x 64] and one x box
//    [NT x 64] per 64-column slice, 128-byte swizzle).  Warp 1: TMEM owner and
//    MMA issuer.  Warps 2-9: epilogue; warp e = w - 2 reads TMEM lane quadrant
//    q = w % 4 (tile rows 32q..32q+31) in accumulator columns
//    [h HALF, (h+1) HALF), h = e / 4, HALF = G NT / 2.
//  * A whole group is stored straight from TMEM.  A split group is reduced by
//    a reduce-scatter among the blocks that touch it: its eligible reducers
//    are the contributors that visit it last (every contributor except the
//    first one when that one's range starts in an earlier group); each takes a
//    contiguous share of the 8 column blocks (HALF / 8 accumulator columns
//    each).  A contributor publishes every column block it does not reduce as
//    plain FP32 (float4 stores, layout [column / 4][lane][4] per warp chunk),
//    fences, and sets one flag per consumer.  A reducer waits for the flags
//    (bounded), copies the other contributors' column blocks into its idle
//    shared-memory ring with bulk copies, adds every contributor's value in
//    increasing block order (its own from TMEM), rounds to BF16, stores y and
//    clears the flags it consumed.  Every block publishes all it owes before
//    it waits on anything, so no wait depends on a waiting block; the split
//    reads are spread over the contributors instead of one block per group.
//    No float atomics: results are identical from run to run.
//  * Every wait is bounded in time; on a give-up the block records a code,
//    lets every role finish, waits for its MMAs and copies, and frees TMEM.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace dep {
namespace {

constexpr int kBM = 128;           // weight rows per tile (MMA M)
constexpr int kBK = 64;            // columns per slice: one 128-byte swizzle row
constexpr int kUmmaK = 16;         // K of one kind::f16 MMA
constexpr int kEpiWarps = 8;       // two per TMEM lane quadrant
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kWBytes = kBM * kBK * 2;  // one weight slice: 16 KB
constexpr int kColBlocks = 8;      // reduce-scatter granularity per warp chunk (at most)
constexpr int kMaxStaging = 8;     // staging buffers per reducing warp

template <int NT, int G>
struct WideShape {
    static constexpr int ROWS = G * kBM;               // weight rows per group
    static constexpr int ACC = G * NT;                 // TMEM columns of one accumulator
    static constexpr int BUFS = 2 * ACC <= 512 ? 2 : 1;
    static constexpr uint32_t TMEM_COLS = BUFS * ACC;  // a power of two >= 64
    static constexpr int HALF = ACC / 2;               // accumulator columns per epilogue warp
    static constexpr int CBW = HALF / kColBlocks >= 16 ? HALF / kColBlocks : 16;  // columns per block
    static constexpr int NCB = HALF / CBW;             // column blocks per warp chunk (<= 8)
    static constexpr int CB_FLOATS = 32 * CBW;         // one column block of a warp chunk
    static constexpr int CHUNK = 32 * HALF;            // floats of one warp chunk
    static constexpr int PIECE = kEpiWarps * CHUNK;    // floats of one block's piece (ROWS x NT)
    static constexpr int X_BYTES = NT * kBK * 2;
    static constexpr int ATOM = G * kWBytes + X_BYTES;  // bytes per 64-column slice
    static_assert(ACC <= 512 && NT >= 32 && NT <= 256 && (G == 2 || G == 4), "shape");
    static_assert(CBW % 16 == 0 && NT % CBW == 0 && NCB <= kColBlocks, "column blocks");
    static_assert(PIECE == ROWS * NT, "piece layout");
};

__device__ __forceinline__ uint16_t to_bf16(float v)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ int ld_acquire(const int *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed(int *p, int v)
{
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Later bulk (async-proxy) reads of global memory see what generic stores made
// visible before it.
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// The split of one group among the blocks of a stream-K launch.
struct GroupSplit {
    int64_t c_a, c_b;  // first and last contributor
    int64_t c_e;       // first eligible reducer (contributors c_e..c_b visit the group last)
    __device__ GroupSplit(int64_t t, int64_t KT, int64_t U, int64_t C)
    {
        c_a = sk_owner(t * KT, U, C);
        c_b = sk_owner(t * KT + KT - 1, U, C);
        c_e = c_a + (sk_begin(c_a, U, C) < t * KT ? 1 : 0);
    }
    __device__ bool split() const { return c_a != c_b; }
    __device__ int64_t reducers() const { return c_b - c_e + 1; }
    // Column blocks [cb_begin(i), cb_begin(i + 1)) are reduced by reducer c_e + i.
    __device__ int cb_begin(int64_t i, int ncb) const { return (int)((i * ncb) / reducers()); }
    // Index (from c_e) of the reducer whose share holds column block cb: the
    // largest i with cb_begin(i) <= cb.
    __device__ int64_t reducer_index(int cb, int ncb) const
    {
        const int64_t r = reducers(), i = (((int64_t)cb + 1) * r - 1) / ncb;
        return i < r - 1 ? i : r - 1;
    }
};

// Visit order of a block's groups: its last group, the whole groups in
// between, then its first group (which it may reduce, with the ring idle).
struct WideOrder {
    int64_t u_begin, u_end, kt, t_first, t_last, m;
    __device__ WideOrder(int64_t ub, int64_t ue, int64_t KT)
        : u_begin(ub), u_end(ue), kt(KT), t_first(ub / KT), t_last(ue > ub ? (ue - 1) / KT : ub / KT),
          m(ue > ub ? t_last - t_first + 1 : 0)
    {
    }
    __device__ int64_t tile(int64_t i) const
    {
        if (m == 1)
            return t_first;
        return i == 0 ? t_last : (i == m - 1 ? t_first : t_first + i);
    }
    __device__ int64_t seg_begin(int64_t t) const { return u_begin > t * kt ? u_begin : t * kt; }
    __device__ int64_t seg_end(int64_t t) const { return u_end < (t + 1) * kt ? u_end : (t + 1) * kt; }
    // Workspace slot of the block's piece of group t: 1 for the group it visits
    // last (its first group), 0 for its last group when it has more than one.
    __device__ int slot(int64_t t) const { return t == t_first ? 1 : 0; }
};

__device__ __forceinline__ int slot_of(int64_t c, int64_t t, int64_t KT, int64_t U, int64_t C)
{
    return t == sk_begin(c, U, C) / KT ? 1 : 0;
}

template <int NT, int G>
__global__ void __launch_bounds__(kThreads, 1)
    tc_wide_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   uint16_t *__restrict__ y, int B, int N, int K, int stages, int atoms,
                   float *__restrict__ ws, int *__restrict__ flags, int keep_own, int *__restrict__ status,
                   const Bounds bd, uint64_t limit_ns)
{
    using S = WideShape<NT, G>;
    const int STAGE = atoms * S::ATOM;
    const int KG = atoms * kBK;  // columns per unit
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle tiles need 1 KB alignment
    uint8_t *smem = smem_raw + (base - raw);
    const int RING = stages * STAGE;
    if (!dbg_ok((base - raw) + (size_t)RING + (2 * (size_t)stages + 5 + kEpiWarps * kMaxStaging) * 8 + 8 - 1, bd.smem,
                status))
        return;  // the ring, the barriers and the TMEM slot must lie in the launch's shared memory
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)RING);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = full0 + 8 * stages;
    const uint32_t accf0 = empty0 + 8 * stages;  // accumulator final, 2 buffers
    const uint32_t acce0 = accf0 + 16;           // accumulator drained, 2 buffers
    const uint32_t done = acce0 + 16;            // all MMAs complete
    const uint32_t stg0 = done + 8;              // staging buffers: [warp][kMaxStaging]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * stages + 5 + kEpiWarps * kMaxStaging);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int64_t T = (N + S::ROWS - 1) / S::ROWS, KTILES = (K + KG - 1) / KG, U = T * KTILES;
    const int64_t C = gridDim.x, c = blockIdx.x;
    const int64_t u_begin = sk_begin(c, U, C), u_end = sk_begin(c + 1, U, C);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const WideOrder order(u_begin, u_end, KTILES);

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, kEpiWarps);
        }
        mbar_init(done, 1);
        for (int i = 0; i < kEpiWarps * kMaxStaging; ++i)
            mbar_init(stg0 + 8 * i, 1);
        *abort_flag = 0;
        fence_mbar_init();
        griddep_launch_dependents();
    }
    if (warp == 1) {
        tc::alloc(smem_u32(tmem_slot), S::TMEM_COLS);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            prefetch_tmap(&tmW);
            prefetch_tmap(&tmX);
            const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
            auto issue_w = [&](int st, int64_t u) {
                const int t = (int)(u / KTILES), kg = (int)(u % KTILES);
                const uint32_t sa = base + (uint32_t)(st * STAGE);
                for (int a = 0; a < atoms; ++a)
                    for (int g = 0; g < G; ++g)
                        tma_load_2d(sa + (uint32_t)(a * S::ATOM + g * kWBytes), &tmW, kg * KG + a * kBK,
                                    t * S::ROWS + g * kBM, full0 + 8 * st, pol_w);
            };
            auto issue_x = [&](int st, int64_t u) {
                const int kg = (int)(u % KTILES);
                const uint32_t sa = base + (uint32_t)(st * STAGE);
                for (int a = 0; a < atoms; ++a)
                    tma_load_2d(sa + (uint32_t)(a * S::ATOM + G * kWBytes), &tmX, kg * KG + a * kBK, 0,
                                full0 + 8 * st, pol_x);
            };
            // Units in visit order: segment by segment, increasing k inside each.
            int64_t seg = 0, u = order.m > 0 ? order.seg_begin(order.tile(0)) : 0;
            int64_t u_stop = order.m > 0 ? order.seg_end(order.tile(0)) : 0;
            auto advance = [&]() {
                if (++u < u_stop)
                    return;
                if (++seg < order.m) {
                    u = order.seg_begin(order.tile(seg));
                    u_stop = order.seg_end(order.tile(seg));
                }
            };
            // The weight is not written by preceding work: fill the ring with its
            // first tiles, then wait for the preceding grid before reading x.
            const int64_t total = u_end - u_begin;
            const int64_t pre = total < stages ? total : stages;
            int64_t pre_u[16];
            for (int64_t i = 0; i < pre; ++i, advance()) {
                pre_u[i] = u;
                mbar_arrive_expect_tx(full0 + 8 * (int)i, (uint32_t)STAGE);
                issue_w((int)i, u);
            }
            griddep_wait();
            for (int64_t i = 0; i < pre; ++i)
                issue_x((int)i, pre_u[i]);
            int s = (int)(pre % stages);
            uint32_t ph = pre == stages ? 1u : 0u;
            int64_t issued = pre;
            for (; seg < order.m; advance()) {
                if (*abort_flag)
                    break;
                if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, limit_ns)) {
                    record_status(status, DEP_DEV_TIMEOUT_PRODUCER);
                    *abort_flag = 1;
                    break;
                }
                mbar_arrive_expect_tx(full0 + 8 * s, (uint32_t)STAGE);
                issue_w(s, u);
                issue_x(s, u);
                ++issued;
                if (++s == stages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            const int64_t n = issued < stages ? issued : stages;  // drain copies in flight
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
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, NT);
            int s = 0, buf = 0;
            uint32_t ph = 0, acce_ph = 0;
            bool ok = true;
            for (int64_t seg = 0; seg < order.m && ok; ++seg) {
                const int64_t t = order.tile(seg);
                const int64_t sb = order.seg_begin(t), se = order.seg_end(t);
                if (!mbar_wait(acce0 + 8 * buf, ((acce_ph >> buf) & 1u) ^ 1u, limit_ns)) {
                    record_status(status, DEP_DEV_TIMEOUT_MMA);
                    *abort_flag = 1;
                    break;
                }
                acce_ph ^= 1u << buf;
                tc::fence_after();
                const uint32_t d = tmem + (uint32_t)(buf * S::ACC);
                for (int64_t u = sb; u < se; ++u) {
                    if (*abort_flag) {
                        ok = false;
                        break;
                    }
                    if (!mbar_wait(full0 + 8 * s, ph, limit_ns)) {
                        record_status(status, DEP_DEV_TIMEOUT_MMA);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const uint32_t st = base + (uint32_t)(s * STAGE);
                    for (int a = 0; a < atoms; ++a) {
                        const uint32_t sa = st + (uint32_t)(a * S::ATOM);
                        const uint64_t bd = tc::desc_sw128(sa + (uint32_t)(G * kWBytes));
#pragma unroll
                        for (int j = 0; j < kBK / kUmmaK; ++j) {
                            // advance along K inside the 128-byte swizzle row: 32 bytes per step
                            const uint64_t off = (uint64_t)((j * kUmmaK * 2) >> 4);
                            const uint32_t acc = (u != sb || a > 0 || j > 0) ? 1u : 0u;
#pragma unroll
                            for (int g = 0; g < G; ++g)
                                tc::mma_bf16(d + (uint32_t)(g * NT), tc::desc_sw128(sa + (uint32_t)(g * kWBytes)) + off,
                                             bd + off, idesc, acc);
                        }
                    }
                    tc::commit(empty0 + 8 * s);  // the stage is free once these MMAs finish
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok)
                    break;
                tc::commit(accf0 + 8 * buf);  // the accumulator is final
                if (S::BUFS == 2)
                    buf ^= 1;
            }
            tc::commit(done);  // TMEM is freed at the end: wait for every MMA
            if (!mbar_wait(done, 0, limit_ns))
                record_status(status, DEP_DEV_TIMEOUT_MMA);
        }
    } else {
        // ---------------- epilogue warps ----------------
        griddep_wait();  // the workspace, flags and y may still be in use by the preceding grid
        const int e = warp - 2;           // chunk index within a piece
        const int q = warp & 3;           // TMEM lane quadrant this warp may access
        const int h = e >> 2;             // accumulator column half
        const int row = 32 * q + lane;    // row within a tile
        float *const slots = ws;          // [block][slot][PIECE]
        auto chunk = [&](int64_t blk, int sl) -> float * {
            return slots + ((size_t)blk * 2 + sl) * S::PIECE + (size_t)e * S::CHUNK;
        };
        // Flag of (publisher, slot, chunk, consumer column block); one writer, one reader.
        auto flag = [&](int64_t blk, int sl, int cb) -> int * {
            return flags + ((blk * 2 + sl) * kEpiWarps + e) * kColBlocks + cb;
        };
        uint32_t accf_ph = 0;
        int buf = 0;
        // Staging ring of this warp inside the (then idle) weight ring.
        const int stg_bytes = S::CB_FLOATS * 4;
        const int per_warp = (RING / kEpiWarps) / stg_bytes;
        const int n_stg = per_warp < kMaxStaging ? per_warp : kMaxStaging;
        const uint32_t stg_base = base + (uint32_t)(e * (RING / kEpiWarps));
        uint32_t stg_ph = 0;  // parity per staging buffer (bit i)
        for (int64_t seg = 0; seg < order.m; ++seg) {
            const int64_t t = order.tile(seg);
            const bool whole = order.seg_begin(t) == t * KTILES && order.seg_end(t) == (t + 1) * KTILES;
            if (!mbar_wait(accf0 + 8 * buf, (accf_ph >> buf) & 1u, limit_ns)) {
                record_status(status, DEP_DEV_TIMEOUT_EPILOGUE);
                *abort_flag = 1;
                break;
            }
            accf_ph ^= 1u << buf;
            tc::fence_after();
            const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * S::ACC + h * S::HALF);
            // Column block cb covers accumulator columns h HALF + cb CBW ..: tile g, batch b0.
            auto col_tile = [&](int cb) { return (h * S::HALF + cb * S::CBW) / NT; };
            auto col_b0 = [&](int cb) { return (h * S::HALF + cb * S::CBW) % NT; };
            if (whole) {
#pragma unroll 1
                for (int cb = 0; cb < S::NCB; ++cb) {
                    const int b0 = col_b0(cb);
                    if (b0 >= B)
                        continue;
                    const int64_t n = t * S::ROWS + (int64_t)col_tile(cb) * kBM + row;
#pragma unroll 1
                    for (int c16 = 0; c16 < S::CBW; c16 += 16) {
                        __syncwarp();  // tcgen05.ld is warp-collective: every lane, converged
                        uint32_t v[16];
                        tc::ld16(tq + (uint32_t)(cb * S::CBW + c16), v);
                        tc::wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (b0 + c16 + j < B && n < N && dbg_ok((int64_t)(b0 + c16 + j) * N + n, bd.y, status))
                                y[(int64_t)(b0 + c16 + j) * N + n] = to_bf16(__uint_as_float(v[j]));
                    }
                }
            } else {
                const GroupSplit gs(t, KTILES, U, C);
                const int sl = order.slot(t);
                // This block reduces column blocks [my0, my1) of its chunk (empty if
                // it is not an eligible reducer of t, or if there are more reducers
                // than column blocks and its share is empty).
                int my0 = 0, my1 = 0;
                if (c >= gs.c_e) {
                    my0 = gs.cb_begin(c - gs.c_e, S::NCB);
                    my1 = gs.cb_begin(c - gs.c_e + 1, S::NCB);
                }
                // 1. Publish every column block this block does not reduce (all of
                //    them when the pieces are kept for inspection).
#pragma unroll 1
                for (int cb = 0; cb < S::NCB; ++cb) {
                    if (col_b0(cb) >= B || (cb >= my0 && cb < my1 && !keep_own))
                        continue;
                    if (!dbg_range((chunk(c, sl) - ws) + (size_t)cb * S::CB_FLOATS, S::CB_FLOATS, bd.ws, status))
                        continue;
                    float4 *dst = reinterpret_cast<float4 *>(chunk(c, sl) + (size_t)cb * S::CB_FLOATS);
#pragma unroll 1
                    for (int c16 = 0; c16 < S::CBW; c16 += 16) {
                        __syncwarp();  // tcgen05.ld is warp-collective: every lane, converged
                        uint32_t v[16];
                        tc::ld16(tq + (uint32_t)(cb * S::CBW + c16), v);
                        tc::wait_ld();
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[(c16 / 4 + i) * 32 + lane] =
                                make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                            __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                    }
                }
                __threadfence();
                __syncwarp();
                // One flag per consumer: lane cb < NCB signals the reducer whose share
                // starts at column block cb, unless that reducer is this block.
                if (lane < S::NCB) {
                    const int64_t i = gs.reducer_index(lane, S::NCB);
                    if (gs.cb_begin(i, S::NCB) == lane && gs.c_e + i != c &&
                        dbg_ok(flag(c, sl, lane) - flags, bd.counters, status)) {
                        __threadfence();
                        st_relaxed(flag(c, sl, lane), 1);
                    }
                }
                // 2. Reduce this block's share: every contributor's value in
                //    increasing block order, this block's own from TMEM.
                if (my1 > my0) {
                    bool ok = true;
                    const uint64_t t0 = globaltimer_ns();
                    for (int64_t p = gs.c_a; p <= gs.c_b && ok; ++p) {
                        if (p == c)
                            continue;
                        const int *f = flag(p, slot_of(p, t, KTILES, U, C), my0);
                        if (!dbg_ok(f - flags, bd.counters, status)) {
                            ok = false;
                            break;
                        }
                        while (ld_acquire(f) == 0)
                            if (globaltimer_ns() - t0 > limit_ns) {
                                record_status(status, DEP_DEV_TIMEOUT_EPILOGUE);
                                ok = false;
                                break;
                            }
                    }
                    ok = __all_sync(0xffffffffu, ok);
                    // Copies in consumption order: (valid column block, other
                    // contributor in block order); n_stg of them in flight.
                    const int64_t others = gs.c_b - gs.c_a;
                    int n_valid = 0;
                    for (int cb = my0; cb < my1; ++cb)
                        n_valid += col_b0(cb) < B ? 1 : 0;
                    const int64_t n_copy = (int64_t)n_valid * others;
                    auto copy_src = [&](int64_t i) -> const float * {
                        int64_t k = i / others, j = i % others;
                        int cb = my0;
                        for (;; ++cb)
                            if (col_b0(cb) < B && k-- == 0)
                                break;
                        int64_t p = gs.c_a + j;
                        if (p >= c)
                            ++p;
                        return chunk(p, slot_of(p, t, KTILES, U, C)) + (size_t)cb * S::CB_FLOATS;
                    };
                    auto issue = [&](int64_t i) {
                        const int sb = (int)(i % n_stg);
                        const uint32_t bar = stg0 + 8 * (e * kMaxStaging + sb);
                        const float *src = copy_src(i);
                        mbar_arrive_expect_tx(bar, (uint32_t)stg_bytes);
                        if (dbg_range(src - ws, S::CB_FLOATS, bd.ws, status) &&
                            dbg_range((stg_base - base) + (uint32_t)(sb * stg_bytes), stg_bytes, (uint32_t)RING, status))
                            bulk_load(stg_base + (uint32_t)(sb * stg_bytes), src, (uint32_t)stg_bytes, bar);
                    };
                    int64_t issued = 0, used = 0;
                    if (ok && lane == 0) {
                        fence_proxy_async_global();  // the bulk copies read what the flags published
                        for (; issued < n_copy && issued < n_stg; ++issued)
                            issue(issued);
                    }
                    issued = __shfl_sync(0xffffffffu, issued, 0);
#pragma unroll 1
                    for (int cb = my0; cb < my1 && ok; ++cb) {
                        const int b0 = col_b0(cb);
                        if (b0 >= B)
                            continue;
                        const int64_t n = t * S::ROWS + (int64_t)col_tile(cb) * kBM + row;
                        float sum[S::CBW];
#pragma unroll 1
                        for (int64_t p = gs.c_a; p <= gs.c_b && ok; ++p) {
                            float v[S::CBW];
                            if (p == c) {
#pragma unroll
                                for (int c16 = 0; c16 < S::CBW; c16 += 16) {
                                    __syncwarp();
                                    uint32_t o[16];
                                    tc::ld16(tq + (uint32_t)(cb * S::CBW + c16), o);
                                    tc::wait_ld();
#pragma unroll
                                    for (int j = 0; j < 16; ++j)
                                        v[c16 + j] = __uint_as_float(o[j]);
                                }
                            } else {
                                const int sb = (int)(used % n_stg);
                                if (!mbar_wait(stg0 + 8 * (e * kMaxStaging + sb), (stg_ph >> sb) & 1u, limit_ns)) {
                                    record_status(status, DEP_DEV_TIMEOUT_EPILOGUE);
                                    ok = false;
                                }
                                ok = __all_sync(0xffffffffu, ok);
                                if (!ok)
                                    break;
                                const float4 *src = reinterpret_cast<const float4 *>(
                                    smem + (stg_base - base) + (size_t)sb * stg_bytes);
#pragma unroll
                                for (int i = 0; i < S::CBW / 4; ++i) {
                                    const float4 f = src[i * 32 + lane];
                                    v[4 * i] = f.x;
                                    v[4 * i + 1] = f.y;
                                    v[4 * i + 2] = f.z;
                                    v[4 * i + 3] = f.w;
                                }
                                stg_ph ^= 1u << sb;
                                ++used;
                                __syncwarp();  // every lane has read the buffer: refill it
                                if (lane == 0 && issued < n_copy)
                                    issue(issued);
                                ++issued;
                            }
#pragma unroll
                            for (int j = 0; j < S::CBW; ++j)
                                sum[j] = p == gs.c_a ? v[j] : sum[j] + v[j];
                        }
                        if (!ok)
                            break;
#pragma unroll
                        for (int j = 0; j < S::CBW; ++j)
                            if (b0 + j < B && n < N && dbg_ok((int64_t)(b0 + j) * N + n, bd.y, status))
                                y[(int64_t)(b0 + j) * N + n] = to_bf16(sum[j]);
                    }
                    if (!ok && lane == 0) {
                        // Let copies still in flight land (bounded) before the block
                        // leaves; nothing reads them.
                        for (int64_t i = used; i < issued && i < n_copy; ++i) {
                            const int sb = (int)(i % n_stg);
                            mbar_wait(stg0 + 8 * (e * kMaxStaging + sb), (stg_ph >> sb) & 1u, limit_ns);
                            stg_ph ^= 1u << sb;
                        }
                    }
                    // The flags this warp consumed are clear for the next launch.
                    __syncwarp();
                    if (lane == 0 && ok)
                        for (int64_t p = gs.c_a; p <= gs.c_b; ++p)
                            if (p != c)
                                st_relaxed(flag(p, slot_of(p, t, KTILES, U, C), my0), 0);
                }
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(acce0 + 8 * buf);
            if (S::BUFS == 2)
                buf ^= 1;
        }
    }

    __syncwarp();
    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after();
        tc::dealloc(tmem, S::TMEM_COLS);
    }
}

// Shared memory after the 1 KB-aligned ring: full[stages], empty[stages],
// accf[2], acce[2], done, the staging barriers; then the TMEM address and the
// abort flag.  Launches ask for at least half of an SM's shared memory, so a
// block never shares its SM (and its TMEM) with another block of this kernel.
size_t smem_bytes_of(int stages, int atoms, int atom_bytes)
{
    const size_t need = 1024 + (size_t)stages * atoms * atom_bytes +
                        (size_t)(2 * stages + 5 + kEpiWarps * kMaxStaging) * 8 + 16;
    const size_t floor_b = (size_t)kMaxDynamicSmem / 2 + 1024;
    return need > floor_b ? need : floor_b;
}

template <int NT, int G>
size_t smem_bytes(int stages, int atoms)
{
    return smem_bytes_of(stages, atoms, WideShape<NT, G>::ATOM);
}

template <int NT, int G>
cudaError_t prepare()
{
    static std::atomic<uint64_t> devices{0};
    return set_smem_attr(tc_wide_kernel<NT, G>, devices);
}

int64_t groups_of(const dep_tactic_t &t, int64_t N) { return (N + t.tile_n - 1) / t.tile_n; }

int64_t units_of(const dep_tactic_t &t, int64_t N, int64_t K)
{
    return groups_of(t, N) * ((K + t.tile_k - 1) / t.tile_k);
}

template <int NT, int G>
cudaError_t run_shape(const dep_tactic_t &t, const RunArgs &a)
{
    cudaError_t e = prepare<NT, G>();
    if (e != cudaSuccess)
        return e;
    CUtensorMap tmW, tmX;
    if (encode_bf16_2d(&tmW, a.W, (uint64_t)a.K, (uint64_t)a.N, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B) !=
        CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int atoms = t.tile_k / kBK;
    const int64_t U = units_of(t, a.N, a.K);
    const int grid = (int)(U < t.ctas ? U : t.ctas);
    const size_t smem = smem_bytes<NT, G>(t.stages, atoms);
    for (int32_t r0 = 0; r0 < a.B; r0 += NT) {
        const int32_t rows = a.B - r0 < NT ? a.B - r0 : NT;
        if (encode_bf16_2d(&tmX, a.x + (size_t)r0 * a.K, (uint64_t)a.K, (uint64_t)rows, kBK, NT,
                           CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        e = launch(tc_wide_kernel<NT, G>, dim3(grid), dim3(kThreads), smem, a.stream, a.pdl, tmW, tmX,
                   a.y + (size_t)r0 * a.N, rows, (int)a.N, (int)a.K, t.stages, atoms, a.ws, a.counters,
                   a.keep_pieces ? 1 : 0, a.status, a.bounds(rows, smem), a.wait_limit_ns);
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

template <int NT, int G>
int blocks_per_sm_shape(const dep_tactic_t &t)
{
    if (prepare<NT, G>() != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, tc_wide_kernel<NT, G>, kThreads,
                                                      smem_bytes<NT, G>(t.stages, t.tile_k / kBK)) != cudaSuccess)
        return 0;
    return n;
}

template <int NT, int G>
size_t smem_shape(const dep_tactic_t &t)
{
    return smem_bytes<NT, G>(t.stages, t.tile_k / kBK);
}

template <int NT, int G>
cudaError_t prepare_shape(const dep_tactic_t &)
{
    return prepare<NT, G>();
}

template <int NT, int G>
size_t piece_floats(const dep_tactic_t &)
{
    return (size_t)WideShape<NT, G>::PIECE;
}

// The instantiation of a tactic: MMA width (cols) x tiles per group (tile_n / 128).
#define DEP_WIDE_DISPATCH(NAME, RET, FN, BAD)                                   \
    RET NAME(const dep_tactic_t &t)                                             \
    {                                                                           \
        const int g = t.tile_n / kBM;                                           \
        switch (t.cols) {                                                       \
        case 32: return g == 4 ? FN<32, 4>(t) : g == 2 ? FN<32, 2>(t) : BAD;    \
        case 64: return g == 4 ? FN<64, 4>(t) : g == 2 ? FN<64, 2>(t) : BAD;    \
        case 128: return g == 4 ? FN<128, 4>(t) : g == 2 ? FN<128, 2>(t) : BAD; \
        case 256: return g == 2 ? FN<256, 2>(t) : BAD;                          \
        default: return BAD;                                                    \
        }                                                                       \
    }

DEP_WIDE_DISPATCH(smem_for, size_t, smem_shape, 0)
DEP_WIDE_DISPATCH(blocks_for, int, blocks_per_sm_shape, 0)
DEP_WIDE_DISPATCH(prepare_for, cudaError_t, prepare_shape, cudaErrorInvalidValue)
DEP_WIDE_DISPATCH(piece_for, size_t, piece_floats, 0)
#undef DEP_WIDE_DISPATCH

}  // namespace

bool wide_valid(const dep_tactic_t &t)
{
    if (t.kind != DEP_KIND_TC_WIDE || t.ctas < 1 || (t.tile_n != 2 * kBM && t.tile_n != 4 * kBM))
        return false;
    if (t.tile_k != kBK && t.tile_k != 2 * kBK)
        return false;  // 1 or 2 slices of 64 columns per stage
    if (t.stages < 2 || t.stages > 16 || t.splits != 0)
        return false;
    const size_t smem = smem_for(t);
    return smem != 0 && smem <= (size_t)kMaxDynamicSmem;
}

int64_t wide_units(const dep_tactic_t &t, int64_t N, int64_t K) { return units_of(t, N, K); }

size_t wide_ws_per_cta(const dep_tactic_t &t) { return 2 * piece_for(t); }  // two slots per block

size_t wide_flags_per_cta(const dep_tactic_t &) { return (size_t)2 * kEpiWarps * kColBlocks; }

int wide_blocks_per_sm(const dep_tactic_t &t) { return blocks_for(t); }

cudaError_t wide_prepare_device()
{
    for (int32_t cols : {32, 64, 128, 256})
        for (int32_t g : {2, 4}) {
            if (cols * g > 512)
                continue;
            dep_tactic_t t{};
            t.cols = cols;
            t.tile_n = g * kBM;
            const cudaError_t e = prepare_for(t);
            if (e != cudaSuccess)
                return e;
        }
    return cudaSuccess;
}

cudaError_t wide_run(const dep_tactic_t &t, const RunArgs &a)
{
    const int g = t.tile_n / kBM;
    switch (t.cols) {
    case 32: return g == 4 ? run_shape<32, 4>(t, a) : run_shape<32, 2>(t, a);
    case 64: return g == 4 ? run_shape<64, 4>(t, a) : run_shape<64, 2>(t, a);
    case 128: return g == 4 ? run_shape<128, 4>(t, a) : run_shape<128, 2>(t, a);
    case 256: return run_shape<256, 2>(t, a);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace dep
