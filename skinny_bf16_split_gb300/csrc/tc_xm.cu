// tc_xm.cu -- tcgen05 tactic for wide batches with x on the MMA's M side.
//
// Computes y[B,N] = BF16(x[B,K] . W[N,K]^T), BF16 products accumulated in FP32,
// for the batches past the split-K rows (runtime.hybrid page,
// HybridAttention.__init__: past them the projection runs the stock
// FP32-accumulated BF16 GEMM; runtime.dep page, DepProjection.run).
//
// Why: the other tensor-core kinds put 128 weight rows on the MMA's M side and
// the batch on N (swap-AB).  A tile of 128 weight rows is the smallest M that
// runs at the full MMA rate, so a 14560-row weight makes 114 tiles for 152 SMs,
// and at 64-256 batch rows the tiles must be grouped and split along K (the
// cluster kind), or a 64-row tile half wastes the tensor pipe.  Here the roles
// are the other way round: the batch rows are the M side (x is operand A), a
// tile of R weight rows is the N side (W is operand B), and R -- any multiple
// of 16 up to 256 -- is chosen so that the tiles nearly fill the SMs (DSA:
// R = 96, 152 tiles).  Every block streams its tiles' whole K: no K split, no
// partials, no exchange, no cluster.
//
// Design (sm_103a, one CTA per SM, no multicast):
//  * Tiles of R weight rows are dealt out statically: block b takes tiles
//    b, b + grid, ...
//  * A stage holds `atoms` 64-column slices of the tile's weight rows [R x 64]
//    side by side (each weight row read in runs of 128 x atoms contiguous
//    bytes), then the same slices of x: MB blocks (one or two) of MR batch rows,
//    MR = the MMA's M: 128, or 64 for a pass of at most 64 rows (the MMA costs
//    the same, and x takes half the shared memory).  The weight is one copy per
//    stage and x one per block, through column-block views when K % 64 == 0;
//    one copy per slice otherwise.  Rows past the pass and columns past K read
//    as zero.
//  * Warp 0 lane 0: TMA producer.  With programmatic dependent launch it fills
//    the first stages' weight before waiting for the preceding grid (the weight
//    is never written by preceding work) and loads x only after it.
//  * Warps 1 and 2 lane 0: MMA issuers (K = 16 per MMA), each into its own
//    accumulator.  One thread issues an MMA only every ~45-120 cycles, which at
//    N = R would not keep up with the weight stream, so two issue: with one
//    block of batch rows (MB = 1) issuer i takes K steps 2i and 2i + 1 of every
//    slice and the epilogue adds the two accumulators (issuer 0's first); with
//    two blocks (MB = 2) issuer i takes block i.  Warp 1 owns TMEM.  Two
//    accumulator buffers of 2 R columns where they fit, so the epilogue of a
//    tile overlaps the next tile's MMAs.
//  * Warps 3-10: epilogue.  Two warps per TMEM lane quadrant take alternate
//    16-column chunks (= 16 consecutive weight rows), round to BF16 and store
//    32 contiguous bytes of a y row per lane.  M = 128 puts batch row r in
//    TMEM lane r; M = 64 puts it in lane 32 (r / 16) + r % 16.
//  * Pairs (splits = 2): where x's bytes per step would outweigh the weight's
//    at tiles that fill the SMs, a thread-block cluster of two CTAs shares each
//    tile of up to twice the rows, rank r summing the first or second half of
//    the 64-column slices.  Once its MMAs of the tile are done a CTA's ring is
//    idle: it arms a barrier with the bytes to come, tells the other CTA, sends
//    the other CTA's half of its accumulator columns into that CTA's ring
//    (st.async, counted on its barrier), waits for its own half, adds the two K
//    halves (rank 0's first) and stores its half of the tile's y.  The producer
//    refills the ring for the next tile only after the epilogue is done with
//    the received partials.  Cluster barriers after set-up and before exit.
//  * Batches wider than 128 MB rows run in passes.
//  * Every wait on a barrier is bounded in time; on a give-up the block records
//    a code, lets every role stop, waits for its own copies and MMAs, and frees
//    TMEM.  Every output is the FP32 sum of fixed MMA accumulation chains over K
//    in increasing order: results do not depend on the grid or on timing.
#include <cuda_bf16.h>

#include "cluster.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace dep {
namespace {

constexpr int kBK = 64;          // columns per slice: one 128-byte swizzle row
constexpr int kXRows = 128;      // batch rows per block of x
constexpr int kIssuers = 2;      // warps 1 and 2
constexpr int kEpi0 = 3;         // first epilogue warp
constexpr int kEpiWarps = 8;     // two per TMEM lane quadrant
constexpr int kThreads = 32 * (kEpi0 + kEpiWarps);
constexpr int kMaxRows = 256;    // MMA N limit (and TMA box limit)
constexpr int kMaxStages = 16;

// One stage: `atoms` weight slices of R rows, then MB blocks of `atoms` x slices of mr rows.
__host__ __device__ constexpr int xm_stage(int atoms, int mb, int R, int mr)
{
    return atoms * (R + mb * mr) * kBK * 2;
}
// TMEM columns of one accumulator buffer: one R-column accumulator per issuer.
__host__ __device__ constexpr int xm_acc(int R) { return kIssuers * R; }
// Accumulator buffers: two when both fit in the 512 TMEM columns.
__host__ __device__ constexpr int xm_bufs(int R) { return 2 * xm_acc(R) <= 512 ? 2 : 1; }
// TMEM columns to allocate: a power of two >= 32.
__host__ __device__ inline uint32_t xm_tmem_cols(int R)
{
    const uint32_t need = (uint32_t)(xm_bufs(R) * xm_acc(R));
    uint32_t c = 32;
    while (c < need)
        c <<= 1;
    return c;
}
// Shared memory: the 1 KB-aligned ring; then full[stages], empty[stages],
// accf[2], acce[2], done, ring_free, rx_full, peer_free; then the TMEM address
// and the abort flag.
__host__ __device__ constexpr size_t xm_smem_bytes(int stages, int atoms, int mb, int R, int mr)
{
    return 1024 + (size_t)stages * xm_stage(atoms, mb, R, mr) + (size_t)(2 * stages + 8) * 8 + 16;
}
// Bytes one CTA of a pair receives from the other: half the R accumulator
// columns of every block of 128 batch rows, FP32 (laid out [block][lane
// quadrant][column / 4][lane][4]).
__host__ __device__ constexpr size_t xm_recv_bytes(int mb, int R) { return (size_t)mb * kXRows * (R / 2) * 4; }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

// Instruction descriptor of kind::f16 (FP32 accumulator, BF16 A and B, both
// K-major) for a runtime M and N.
__device__ __forceinline__ uint32_t idesc_mn(int m, int n)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

template <int MB, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    tc_xm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                 uint16_t *__restrict__ y, int B, int N, int K, int R, int MR, int stages, int atoms, int tma3,
                 int *__restrict__ status, const Bounds bd, uint64_t limit_ns)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle boxes need 1 KB alignment
    uint8_t *smem = smem_raw + (base - raw);
    const int STAGE = xm_stage(atoms, MB, R, MR);
    const int WSLICE = R * kBK * 2, XBOX = MR * kBK * 2;  // one weight slice; one slice of one x block
    const int XOFF = atoms * WSLICE;                      // x after the weight in a stage
    // The ring, the barriers and the TMEM slot must lie in the launch's shared memory.
    if (!dbg_ok((base - raw) + xm_smem_bytes(stages, atoms, MB, R, MR) - 1024 - 1, bd.smem, status))
        return;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)stages * STAGE);
    const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * stages;
    const uint32_t accf0 = empty0 + 8 * stages;  // accumulator final, 2 buffers
    const uint32_t acce0 = accf0 + 16;           // accumulator drained, 2 buffers
    const uint32_t done = acce0 + 16;            // all MMAs complete
    const uint32_t ring_free = done + 8;         // pairs: the epilogue no longer uses the ring
    const uint32_t rx_full = done + 16;          // pairs: the other CTA's partials have landed
    const uint32_t peer_free = done + 24;        // pairs: the other CTA's ring is idle
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * stages + 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int T = (N + R - 1) / R;            // weight tiles
    // A pair (a cluster of two CTAs) shares each tile: rank r sums the 64-column
    // slices [r KT / 2, (r + 1) KT / 2) and the halves meet in shared memory.
    const int rank = PAIR ? (int)cluster_rank() : 0;
    const int KT_ALL = (K + kBK - 1) / kBK;
    const int S0 = PAIR ? rank * KT_ALL / 2 : 0;  // this CTA's first slice
    const int KT = PAIR ? (rank + 1) * KT_ALL / 2 - S0 : KT_ALL;  // its slices of a tile
    // Tiles are dealt out per block, or per pair: t0, t0 + TS, ...
    const int t0 = PAIR ? (int)cluster_id() : (int)blockIdx.x;
    const int TS = PAIR ? (int)cluster_count() : (int)gridDim.x;
    const int KS = (KT + atoms - 1) / atoms;  // stages per tile
    const int ACC = xm_acc(R);                // TMEM columns of one accumulator buffer
    const int BUFS = xm_bufs(R);
    const uint32_t TMEM_COLS = xm_tmem_cols(R);
    // Blocks of batch rows that hold rows of this pass (a pass of B <= 128 rows
    // in a two-block launch loads and multiplies only the first).
    const int MBV = B > kXRows ? MB : 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto slices_of = [&](int k) { return KT - k * atoms < atoms ? KT - k * atoms : atoms; };

    // Producer state (thread 0).
    uint64_t pol_w = 0, pol_x = 0;
    // The bytes a stage's copies bring (weight and x), armed with its weight copy.
    auto stage_bytes = [&](int na) {
        return tma3 ? atoms * (WSLICE + MBV * XBOX) : na * (WSLICE + MBV * XBOX);
    };
    auto issue_w = [&](int st, int t, int k) {
        const uint32_t dst = base + (uint32_t)(st * STAGE), bar = full0 + 8 * st;
        const int na = slices_of(k);
        mbar_arrive_expect_tx(bar, (uint32_t)stage_bytes(na));
        if (tma3) {  // the stage's slices in one copy; blocks past K read as zero
            tma_load_3d(dst, &tmW, 0, t * R, S0 + k * atoms, bar, pol_w);
        } else {
            for (int a = 0; a < na; ++a)
                tma_load_2d(dst + (uint32_t)(a * WSLICE), &tmW, (S0 + k * atoms + a) * kBK, t * R, bar, pol_w);
        }
    };
    auto issue_x = [&](int st, int k) {
        const uint32_t dst = base + (uint32_t)(st * STAGE + XOFF), bar = full0 + 8 * st;
        const int na = slices_of(k);
        for (int m = 0; m < MBV; ++m) {
            if (tma3) {
                tma_load_3d(dst + (uint32_t)(m * atoms * XBOX), &tmX, 0, m * kXRows, S0 + k * atoms, bar, pol_x);
            } else {
                for (int a = 0; a < na; ++a)
                    tma_load_2d(dst + (uint32_t)((m * atoms + a) * XBOX), &tmX, (S0 + k * atoms + a) * kBK, m * kXRows,
                                bar, pol_x);
            }
        }
    };
    const int pre = KS < stages ? KS : stages;  // stages of the first tile filled before the wait

    if (threadIdx.x == 0) {
        for (int i = 0; i < stages; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, kIssuers);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, kIssuers);
            mbar_init(acce0 + 8 * b, kEpiWarps);
        }
        mbar_init(done, kIssuers);
        mbar_init(ring_free, kEpiWarps);
        mbar_init(rx_full, 1);    // armed per tile with the bytes the other CTA stores
        mbar_init(peer_free, 1);  // arrived on by the other CTA
        *abort_flag = 0;
        fence_mbar_init();
        griddep_launch_dependents();
        // The weight is not written by preceding work: fill the ring with the
        // first tile's first weight slices while warp 1 allocates TMEM.
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmX);
        pol_w = policy_evict_first();
        pol_x = policy_evict_last();
        for (int i = 0; i < pre; ++i)
            issue_w(i, t0, i);
    }
    if (warp == 1) {
        tc::alloc(smem_u32(tmem_slot), TMEM_COLS);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (PAIR)
        cluster_sync();  // both CTAs of the pair have set up their barriers
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            griddep_wait();  // x may be written by the preceding grid
            for (int i = 0; i < pre; ++i)
                issue_x(i, i);
            int t = t0, k = pre, s = pre % stages, gi = 0;
            uint32_t ph = pre == stages ? 1u : 0u;
            int64_t issued = pre;
            for (;;) {
                if (k == KS) {  // the tile is fully issued: the next one of this block
                    t += TS;
                    if (t >= T)
                        break;
                    k = 0;
                    // A pair's partials of the previous tile pass through the ring:
                    // refill it once the epilogue is done with them.
                    if (PAIR && !mbar_wait(ring_free, (uint32_t)(gi & 1), limit_ns)) {
                        record_status(status, DEP_DEV_TIMEOUT_PRODUCER);
                        *abort_flag = 1;
                        break;
                    }
                    ++gi;
                }
                if (*abort_flag)
                    break;
                if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, limit_ns)) {
                    record_status(status, DEP_DEV_TIMEOUT_PRODUCER);
                    *abort_flag = 1;
                    break;
                }
                issue_w(s, t, k);
                issue_x(s, k);
                ++k;
                ++issued;
                if (++s == stages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            // Drain: the most recent fills (at most one per stage) land before the
            // block may leave.
            const int64_t n = issued < stages ? issued : stages;
            for (int64_t i = 0; i < n; ++i) {
                if (--s < 0) {
                    s = stages - 1;
                    ph ^= 1u;
                }
                if (!mbar_wait(full0 + 8 * s, ph, limit_ns))
                    record_status(status, DEP_DEV_TIMEOUT_PRODUCER);
            }
        }
    } else if (warp == 1 || warp == 2) {
        // ---------------- MMA issuers ----------------
        // MB = 1: issuer i takes K steps 2i, 2i + 1 of every slice of block 0.
        // MB = 2: issuer i takes every K step of block i (nothing if that block
        // holds no rows of this pass).
        const int i = warp - 1;
        const int m = MB == 1 ? 0 : i;
        const int j0 = MB == 1 ? 2 * i : 0;
        const bool active = m < MBV;
        if (lane == 0) {
            const uint32_t idesc = idesc_mn(MR, R);
            int s = 0, buf = 0;
            uint32_t ph = 0, acce_ph = 0;
            bool ok = true;
            for (int t = t0; t < T && ok; t += TS) {
                if (!mbar_wait(acce0 + 8 * buf, ((acce_ph >> buf) & 1u) ^ 1u, limit_ns)) {
                    record_status(status, DEP_DEV_TIMEOUT_MMA);
                    *abort_flag = 1;
                    break;
                }
                acce_ph ^= 1u << buf;
                tc::fence_after();
                const uint32_t d = tmem + (uint32_t)(buf * ACC + i * R);
                uint32_t accumulate = 0;
                for (int k = 0; k < KS; ++k) {
                    if (*abort_flag || !mbar_wait(full0 + 8 * s, ph, limit_ns)) {
                        if (!*abort_flag)
                            record_status(status, DEP_DEV_TIMEOUT_MMA);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    if (active) {
                        const uint32_t sa = base + (uint32_t)(s * STAGE);
                        const uint64_t bd0 = tc::desc_sw128(sa) + (uint64_t)(2 * j0);
                        const uint64_t ad0 = tc::desc_sw128(sa + (uint32_t)(XOFF + m * atoms * XBOX)) + (uint64_t)(2 * j0);
                        const int na = slices_of(k);
                        for (int a = 0; a < na; ++a) {
                            // slice a; K steps advance 32 bytes inside the 128-byte rows
                            const uint64_t ad = ad0 + (uint64_t)((a * XBOX) >> 4);
                            const uint64_t bw = bd0 + (uint64_t)((a * WSLICE) >> 4);
                            tc::mma_bf16(d, ad, bw, idesc, accumulate);
                            tc::mma_bf16(d, ad + 2, bw + 2, idesc, 1u);
                            if (MB == 2) {
                                tc::mma_bf16(d, ad + 4, bw + 4, idesc, 1u);
                                tc::mma_bf16(d, ad + 6, bw + 6, idesc, 1u);
                            }
                            accumulate = 1;
                        }
                    }
                    tc::commit(empty0 + 8 * s);  // the stage is free once both issuers' MMAs finish
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok)
                    break;
                tc::commit(accf0 + 8 * buf);  // this issuer's accumulator is final
                if (BUFS == 2)
                    buf ^= 1;
            }
            tc::commit(done);  // TMEM is freed at the end: wait for every MMA
            if (!mbar_wait(done, 0, limit_ns))
                record_status(status, DEP_DEV_TIMEOUT_MMA);
        }
    } else {
        // ---------------- epilogue ----------------
        griddep_wait();  // y may still be in use by the preceding grid
        const int q = warp & 3;             // TMEM lane quadrant this warp may read
        const int h = (warp - kEpi0) >> 2;  // which of the two warps of the quadrant
        const int CPB = R / 16;             // 16-column chunks of one accumulator
        const bool vec = (N & 7) == 0;      // y rows are 16-byte multiples: vector stores
        uint32_t accf_ph = 0;
        int buf = 0, gi = 0;
        uint32_t tq = 0;  // this warp's TMEM lanes of the current accumulator buffer
        // This CTA's FP32 partial of block m, accumulator columns col..col+15
        // (one block of rows: issuer 0's accumulator, then issuer 1's added).
        auto partial = [&](int m, int col, float (&f)[16]) {
            __syncwarp();  // tcgen05.ld is warp-collective: every lane, converged
            uint32_t v[16];
            tc::ld16(tq + (uint32_t)(m * R + col), v);
            tc::wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j)
                f[j] = __uint_as_float(v[j]);
            if (MB == 1) {
                tc::ld16(tq + (uint32_t)(R + col), v);
                tc::wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    f[j] = f[j] + __uint_as_float(v[j]);
            }
        };
        // Round and store the sums of block m, weight rows t R + col .. + 15.
        auto store = [&](int m, int col, int t, const float (&f)[16]) {
            // batch row of this lane in the pass (M = 64: lanes 16-31 hold none)
            const int b = m * kXRows + (MR == kXRows ? 32 * q + lane : (lane < 16 ? 16 * q + lane : kXRows));
            const int n0 = t * R + col;  // first weight row of the chunk
            if (b >= B || n0 >= N)
                return;
            uint16_t *yr = y + (int64_t)b * N + n0;
            if (vec && n0 + 16 <= N && dbg_ok((int64_t)b * N + n0 + 15, bd.y, status)) {
                uint4 lo, hi;
                lo.x = pack_bf16x2(f[0], f[1]);
                lo.y = pack_bf16x2(f[2], f[3]);
                lo.z = pack_bf16x2(f[4], f[5]);
                lo.w = pack_bf16x2(f[6], f[7]);
                hi.x = pack_bf16x2(f[8], f[9]);
                hi.y = pack_bf16x2(f[10], f[11]);
                hi.z = pack_bf16x2(f[12], f[13]);
                hi.w = pack_bf16x2(f[14], f[15]);
                reinterpret_cast<uint4 *>(yr)[0] = lo;
                reinterpret_cast<uint4 *>(yr)[1] = hi;
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (n0 + j < N && dbg_ok((int64_t)b * N + n0 + j, bd.y, status))
                        yr[j] = __bfloat16_as_ushort(__float2bfloat16_rn(f[j]));
            }
        };
        for (int t = t0; t < T; t += TS, ++gi) {
            const bool got = mbar_wait(accf0 + 8 * buf, (accf_ph >> buf) & 1u, limit_ns);
            if (!__all_sync(0xffffffffu, got)) {
                record_status(status, DEP_DEV_TIMEOUT_EPILOGUE);
                *abort_flag = 1;
                break;
            }
            accf_ph ^= 1u << buf;
            tc::fence_after();
            tq = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * ACC);
            bool ok = true;
            if (PAIR) {
                // Rank r reduces and stores accumulator columns [r R/2, (r + 1) R/2)
                // of every block; it sends the other half of its partials to the
                // other CTA's (idle) ring and adds the half it receives, rank 0's
                // K half first.
                const int HALF = R / 2, CPH = HALF / 16, NCH = MBV * CPH;
                const int own0 = rank * HALF, oth0 = HALF - own0;
                const uint32_t par = (uint32_t)(gi & 1), other = (uint32_t)(rank ^ 1);
                auto roff = [&](int m, int c) {  // [block][quadrant][column / 4][lane] float4
                    return (uint32_t)((((m * 4 + q) * (HALF / 4) + c / 4) * 32 + lane) * 16);
                };
                // 1. This CTA's MMAs of the tile are done, so its ring is idle: arm
                //    the receive barrier with the bytes the other CTA will store,
                //    then tell it.
                if (warp == kEpi0 && lane == 0) {
                    mbar_arrive_expect_tx(rx_full, (uint32_t)(MBV * kXRows * HALF * 4));
                    mbar_arrive_peer(peer_addr(peer_free, other));
                }
                // 2. The other CTA's half of this CTA's partials into its ring.
                if (!mbar_wait_cluster(peer_free, par, limit_ns)) {
                    record_status(status, DEP_DEV_TIMEOUT_EPILOGUE);
                    ok = false;
                }
                ok = __all_sync(0xffffffffu, ok);
                if (ok) {
                    const uint32_t pbar = peer_addr(rx_full, other), pbase = peer_addr(base, other);
                    for (int c = h; c < NCH; c += 2) {
                        const int m = c / CPH, col = (c - m * CPH) * 16;
                        float f[16];
                        partial(m, oth0 + col, f);
                        if (!dbg_range(roff(m, col + 12), 16, (unsigned)(stages * STAGE), status))
                            continue;
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            st_async_peer_v4(pbase + roff(m, col + 4 * i), f[4 * i], f[4 * i + 1], f[4 * i + 2],
                                             f[4 * i + 3], pbar);
                    }
                }
                // 3. The other CTA's half of this CTA's columns has landed.
                if (ok && !mbar_wait_cluster(rx_full, par, limit_ns)) {
                    record_status(status, DEP_DEV_TIMEOUT_EPILOGUE);
                    ok = false;
                }
                ok = __all_sync(0xffffffffu, ok);
                // 4. This CTA's columns: the two K halves in rank order.
                for (int c = h; c < NCH && ok; c += 2) {
                    const int m = c / CPH, col = (c - m * CPH) * 16;
                    float f[16], g[16];
                    partial(m, own0 + col, f);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (dbg_range(roff(m, col + 4 * i), 16, (unsigned)(stages * STAGE), status))
                            r = *reinterpret_cast<const float4 *>(smem + roff(m, col + 4 * i));
                        g[4 * i] = r.x;
                        g[4 * i + 1] = r.y;
                        g[4 * i + 2] = r.z;
                        g[4 * i + 3] = r.w;
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        f[j] = rank == 0 ? f[j] + g[j] : g[j] + f[j];
                    store(m, own0 + col, t, f);
                }
            } else {
                for (int c = h; c < MB * CPB; c += 2) {
                    const int m = c / CPB, col = (c - m * CPB) * 16;
                    if (MB == 2 && m >= MBV)
                        break;  // a block past this pass's rows: nothing was summed into it
                    float f[16];
                    partial(m, col, f);
                    store(m, col, t, f);
                }
            }
            if (!ok)
                *abort_flag = 1;
            // The ring (pairs) and the accumulator buffer are free again.
            tc::fence_before();
            __syncwarp();
            if (lane == 0) {
                if (PAIR)
                    mbar_arrive(ring_free);
                mbar_arrive(acce0 + 8 * buf);
            }
            if (BUFS == 2)
                buf ^= 1;
            if (!ok)
                break;
        }
    }

    __syncwarp();
    tc::fence_before();
    __syncthreads();
    if (PAIR)
        cluster_sync();  // no CTA leaves while the other may still write into it
    if (warp == 1) {
        tc::fence_after();
        tc::dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace
}  // namespace dep

namespace dep {
namespace {

template <int MB, bool PAIR>
cudaError_t prepare()
{
    static std::atomic<uint64_t> devices{0};
    return set_smem_attr(tc_xm_kernel<MB, PAIR>, devices);
}

// Stages of a launch whose x blocks have mr rows: the tactic's (which fit at
// 128 rows); a pass of at most 64 rows (MMA M = 64) takes as many more as fit,
// up to twice as many.
int stages_for(const dep_tactic_t &t, int mr)
{
    const int mb = t.cols / kXRows, atoms = t.tile_k / kBK;
    if (mr == kXRows)
        return t.stages;
    int st = t.stages;
    while (st < 2 * t.stages && st < kMaxStages &&
           xm_smem_bytes(st + 1, atoms, mb, t.tile_n, mr) <= (size_t)kMaxDynamicSmem)
        ++st;
    return st;
}

template <int MB, bool PAIR>
cudaError_t run_mb(const dep_tactic_t &t, const RunArgs &a)
{
    cudaError_t e = prepare<MB, PAIR>();
    if (e != cudaSuccess)
        return e;
    const int R = t.tile_n, atoms = t.tile_k / kBK;
    // One copy per stage of the weight and per block of x (column-block views)
    // when K is a multiple of 64; else one per 64-column slice, whose 2-D maps
    // zero-fill past column K.
    const int tma3 = a.K % kBK == 0;
    CUtensorMap tmW, tmX;
    if ((tma3 ? encode_bf16_3d_blocks(&tmW, a.W, (uint64_t)a.K, (uint64_t)a.N, (uint32_t)R, (uint32_t)atoms)
              : encode_bf16_2d(&tmW, a.W, (uint64_t)a.K, (uint64_t)a.N, kBK, (uint32_t)R,
                               CU_TENSOR_MAP_SWIZZLE_128B)) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int64_t T = (a.N + R - 1) / R;
    // blocks (or pairs of blocks) dealing out the tiles
    const int64_t per = PAIR ? t.ctas / 2 : t.ctas;
    const int units = (int)(T < per ? T : per);
    constexpr int32_t kPass = MB * kXRows;
    for (int32_t r0 = 0; r0 < a.B; r0 += kPass) {
        const int32_t rows = a.B - r0 < kPass ? a.B - r0 : kPass;
        // MMA M = 64 for a pass of at most 64 rows (x blocks of 64 rows), else 128
        const int mr = rows <= 64 ? 64 : kXRows, st = stages_for(t, mr);
        const size_t smem = xm_smem_bytes(st, atoms, MB, R, mr);
        const uint16_t *xr = a.x + (size_t)r0 * a.K;
        if ((tma3 ? encode_bf16_3d_blocks(&tmX, xr, (uint64_t)a.K, (uint64_t)rows, (uint32_t)mr, (uint32_t)atoms)
                  : encode_bf16_2d(&tmX, xr, (uint64_t)a.K, (uint64_t)rows, kBK, (uint32_t)mr,
                                   CU_TENSOR_MAP_SWIZZLE_128B)) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(PAIR ? 2 * units : units));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = a.stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = a.pdl ? 1 : 0;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 2;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = PAIR ? 2 : 1;
        e = cudaLaunchKernelEx(&cfg, tc_xm_kernel<MB, PAIR>, tmW, tmX, a.y + (size_t)r0 * a.N, (int)rows,
                               (int)a.N, (int)a.K, R, mr, st, atoms, tma3, a.status, a.bounds(rows, smem),
                               a.wait_limit_ns);
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

}  // namespace

bool xm_valid(const dep_tactic_t &t)
{
    if (t.kind != DEP_KIND_TC_XM || t.ctas < 1 || t.splits < 0 || t.splits > 2)
        return false;  // splits: 0 or 1 = whole K per block; 2 = a pair of blocks per tile
    if (t.tile_n < 16 || t.tile_n > kMaxRows || t.tile_n % 16 != 0)
        return false;  // MMA N: a multiple of 16 up to 256 weight rows
    if (t.cols != kXRows && t.cols != 2 * kXRows)
        return false;  // one or two blocks of 128 batch rows per pass
    if (t.tile_k != kBK && t.tile_k != 2 * kBK && t.tile_k != 4 * kBK)
        return false;  // 1, 2 or 4 slices of 64 columns per stage
    if (t.stages < 2 || t.stages > kMaxStages)
        return false;
    const int atoms = t.tile_k / kBK, mb = t.cols / kXRows;
    if (t.splits == 2) {
        if (t.tile_n % 32 != 0 || t.ctas < 2)
            return false;  // each CTA of a pair stores whole 16-column chunks of a half tile
        // the other CTA's partials land in the idle ring (at 64-row x blocks the ring is smaller)
        if (xm_recv_bytes(mb, t.tile_n) > (size_t)t.stages * xm_stage(atoms, mb, t.tile_n, 64))
            return false;
    }
    return xm_smem_bytes(t.stages, atoms, mb, t.tile_n, kXRows) <= (size_t)kMaxDynamicSmem;
}

int64_t xm_tiles(const dep_tactic_t &t, int64_t N)
{
    const int64_t T = (N + t.tile_n - 1) / t.tile_n;
    return t.splits == 2 ? 2 * T : T;  // blocks a launch can use
}

int xm_stages_fit(int32_t tile_n, int32_t tile_k, int32_t cols, int mr)
{
    int best = 0;
    for (int st = 2; st <= kMaxStages; ++st)
        if (xm_smem_bytes(st, tile_k / kBK, cols / kXRows, tile_n, mr) <= (size_t)kMaxDynamicSmem)
            best = st;
    return best;
}

cudaError_t xm_prepare_device()
{
    cudaError_t e = prepare<1, false>();
    if (e == cudaSuccess)
        e = prepare<2, false>();
    if (e == cudaSuccess)
        e = prepare<1, true>();
    return e == cudaSuccess ? prepare<2, true>() : e;
}

cudaError_t xm_run(const dep_tactic_t &t, const RunArgs &a)
{
    // A pair splits K in two halves of 64-column slices: with fewer than two
    // slices the tactic runs unsplit.
    const bool pair = t.splits == 2 && (a.K + kBK - 1) / kBK >= 2;
    if (t.cols == kXRows)
        return pair ? run_mb<1, true>(t, a) : run_mb<1, false>(t, a);
    return pair ? run_mb<2, true>(t, a) : run_mb<2, false>(t, a);
}

}  // namespace dep
