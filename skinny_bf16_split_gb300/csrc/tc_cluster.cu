// tc_cluster.cu -- tcgen05 tactic for wide batches: a cluster of blocks per weight group.
//
// Computes y[B,N] = BF16(x[B,K] . W[N,K]^T), BF16 products accumulated in FP32,
// for the batches past the split-K rows (runtime.hybrid page,
// HybridAttention.__init__: past them the projection runs the stock
// FP32-accumulated BF16 GEMM; runtime.dep page, DepProjection.run).
//
// Why: at 32-256 batch rows a block that streams one 128-row weight tile takes
// in NT x 128 B of x for every 16 KB of weight, and what one SM can take in --
// not HBM -- bounds the call.  Streaming G = 2 or 4 tiles against each x slice
// cuts that by G, but then there are fewer groups than SMs and every group must
// be split along K; exchanging those FP32 partials through L2 at the end of
// the call costs more than the split saves.  Here the blocks that share a group
// form one thread-block cluster and exchange through distributed shared
// memory, never through global memory.
//
// Design (sm_103a, one CTA per SM, clusters of k CTAs, no multicast):
//  * Cluster j takes groups j, j + C, j + 2C, ... (C clusters); CTA rank r of a
//    cluster streams K piece r (64-column k-tiles [r KT / k, (r+1) KT / k)) of
//    the group: a weight box [tile rows x 64] per tile and k-tile against one
//    x box [NT x 64], one MMA per tile with the same x descriptor (swap-AB; MMA
//    N = the batch padded to NT).  A group is 2 or 4 tiles of 128 rows (MMA
//    M = 128), or one of 128 and one of 64 rows (M = 64; 192 rows, so that
//    the groups of a 14560-row weight fill 152 SMs in clusters of two).  The
//    group's accumulator is one NT-column TMEM block per tile (tile g at
//    column g NT), two buffers where they fit.
//  * The weight and x have rings of their own, each filled by its own producer
//    warp: the weight ring is as deep as shared memory allows (its latency is
//    HBM's), the x ring only a few stages (x is read from L2).
//  * Once its MMAs of a group are done a CTA's rings are idle, and it tells its
//    peers so.  The accumulator columns of every epilogue warp are cut into
//    column blocks; each rank reduces a contiguous share of them.  Every CTA
//    writes the column blocks of each peer's share into that peer's idle ring
//    (st.async, counted on the peer's barrier), then adds the K
//    pieces of its own share in rank order (its own from TMEM), rounds to BF16
//    and stores y.  Results depend only on k, never on timing.
//  * Warps: 0 weight producer, 1 TMEM owner and MMA issuer, 2-9 epilogue
//    (warp w reads TMEM lane quadrant w % 4, column half (w - 2) / 4), 10 x
//    producer.  A cluster barrier after set-up (before any remote access) and
//    one before exit (no CTA leaves while a peer may still write into it).
//  * Every wait on a barrier is bounded in time; on a give-up the CTA records
//    a code, skips what depends on it, waits for its own copies and MMAs, and
//    frees TMEM.
#include <cuda_bf16.h>

#include "cluster.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace dep {
namespace {

constexpr int kBM = 128;        // weight rows per tile (MMA M)
constexpr int kBK = 64;         // columns per k-tile: one 128-byte swizzle row
constexpr int kUmmaK = 16;      // K of one kind::f16 MMA
constexpr int kEpiWarps = 8;    // two per TMEM lane quadrant
constexpr int kXWarp = 2 + kEpiWarps;
constexpr int kThreads = 32 * (kXWarp + 1);
constexpr int kWBytes = kBM * kBK * 2;  // one weight box: 16 KB
constexpr int kColBlocks = 8;   // column blocks per warp chunk (at most)
constexpr int kMaxCluster = 8;  // portable cluster size
constexpr int kMaxXStages = 4;

// G = 2 or 4: that many 128-row tiles per group.  G = 3 stands for one and a
// half: a 128-row tile and a 64-row tile (MMA M = 64), 192 rows per group.
template <int NT, int G>
struct ClusterShape {
    static constexpr int TILES = G == 3 ? 2 : G;       // MMA tiles per group
    static constexpr int ROWS = G == 3 ? 192 : G * kBM;  // weight rows per group
    static constexpr int ACC = TILES * NT;             // TMEM columns of one accumulator
    static constexpr int BUFS = 2 * ACC <= 512 ? 2 : 1;
    static constexpr uint32_t TMEM_COLS = BUFS * ACC;  // a power of two >= 64
    static constexpr int HALF = ACC / 2;               // accumulator columns per epilogue warp
    static constexpr int CBW = HALF / kColBlocks >= 16 ? HALF / kColBlocks : 16;  // columns per block
    static constexpr int NCB = HALF / CBW;             // column blocks per warp chunk
    static constexpr int CB_BYTES = 32 * CBW * 4;      // one column block of a warp chunk (FP32)
    static constexpr int W_STAGE = G == 3 ? kWBytes + kWBytes / 2 : G * kWBytes;
    static constexpr int X_STAGE = NT * kBK * 2;
    // weight rows a column block of the eight warp chunks covers (G = 3: the
    // 64-row tile has 16 rows per TMEM lane quadrant)
    static constexpr int CB_ROWS = G == 3 ? 192 : 256;
    // rows of tile g, and whether TMEM lane `lane` of a quadrant holds one of them
    __host__ __device__ static constexpr int tile_rows(int g) { return G == 3 && g == 1 ? 64 : kBM; }
    static_assert(ACC <= 512 && NT >= 32 && NT <= 256 && (G == 2 || G == 3 || G == 4), "shape");
    static_assert(CBW % 16 == 0 && NT % CBW == 0 && NCB <= kColBlocks, "column blocks");
};

// Column blocks [share_begin(r), share_begin(r + 1)) of every warp chunk are
// reduced by rank r; a rank receives at most max_share of them from each peer.
__host__ __device__ constexpr int share_begin(int r, int ncb, int k) { return (r * ncb) / k; }
__host__ __device__ constexpr int max_share(int ncb, int k) { return (ncb + k - 1) / k; }

// Bytes a rank receives from its peers: (k - 1) senders x 8 warps x max_share blocks.
__host__ __device__ constexpr size_t recv_bytes(int ncb, int k, int cb_bytes)
{
    return (size_t)(k - 1) * kEpiWarps * max_share(ncb, k) * cb_bytes;
}
// y staging for bulk tensor stores, after the received partials: two buffers
// of [2 column halves][CBW batch rows][128 weight rows] BF16.
__host__ __device__ constexpr size_t stage_offset(int ncb, int k, int cb_bytes)
{
    return (recv_bytes(ncb, k, cb_bytes) + 1023) & ~(size_t)1023;
}
__host__ __device__ constexpr size_t stage_bytes(int cbw) { return (size_t)2 * 2 * cbw * kBM * 2; }

// Shared memory after the 1 KB-aligned rings: w_full[SW], w_empty[SW],
// x_full[SX], x_empty[SX], accf[2], acce[2], done, ring_free, rx_full,
// peer_free[kMaxCluster]; then the TMEM address and the abort flag.
__host__ __device__ constexpr int barrier_count(int sw, int sx) { return 2 * sw + 2 * sx + 8 + kMaxCluster; }

__device__ __forceinline__ uint16_t to_bf16(float v)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// The eight epilogue warps (named barrier 1): synchronise, or agree on a flag.
__device__ __forceinline__ void epi_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
}
__device__ __forceinline__ bool epi_all(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(32 * kEpiWarps)
        : "memory");
    return r != 0;
}
// Bulk tensor store of a shared-memory box to global memory (clipped at the
// tensor's bounds), and its completion groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int32_t c0, int32_t c1)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Generic-proxy writes to shared memory become visible to the bulk copies that follow.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }


template <int NT, int G>
__global__ void __launch_bounds__(kThreads, 1)
    tc_cluster_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmW64,
                      const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
                      const __grid_constant__ CUtensorMap tmY64, uint16_t *__restrict__ y, int B, int N, int K,
                      int SW, int SX, int use_tma_y, int *__restrict__ status, const Bounds bd, uint64_t limit_ns)
{
    using S = ClusterShape<NT, G>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle tiles need 1 KB alignment
    uint8_t *smem = smem_raw + (base - raw);
    const uint32_t xbase = base + (uint32_t)(SW * S::W_STAGE);
    const int RING = SW * S::W_STAGE + SX * S::X_STAGE;
    // The rings, the barriers and the TMEM slot must lie in the launch's shared
    // memory, and the received partials and the y staging in the rings.
    if (!dbg_ok((base - raw) + (size_t)RING + (size_t)barrier_count(SW, SX) * 8 + 8 - 1, bd.smem, status) ||
        !dbg_ok(stage_offset(S::NCB, (int)cluster_size(), S::CB_BYTES) + stage_bytes(S::CBW) - 1, (unsigned)RING,
                status))
        return;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)RING);
    const uint32_t wfull0 = smem_u32(bars), wempty0 = wfull0 + 8 * SW;
    const uint32_t xfull0 = wempty0 + 8 * SW, xempty0 = xfull0 + 8 * SX;
    const uint32_t accf0 = xempty0 + 8 * SX;  // accumulator final, 2 buffers
    const uint32_t acce0 = accf0 + 16;        // accumulator drained, 2 buffers
    const uint32_t done = acce0 + 16;         // all MMAs complete
    const uint32_t ring_free = done + 8;      // the epilogue no longer uses the rings
    const uint32_t rx_full = ring_free + 8;   // every peer's partials have landed
    const uint32_t peer_free0 = rx_full + 8;  // peer r's rings are idle (one per rank)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + barrier_count(SW, SX));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int k = (int)cluster_size(), rank = (int)cluster_rank();
    const int64_t T = (N + S::ROWS - 1) / S::ROWS, KT = (K + kBK - 1) / kBK;
    const int64_t CL = cluster_count(), cl = cluster_id();
    const int kt0 = (int)((rank * KT) / k), kt1 = (int)(((rank + 1) * KT) / k);  // this rank's K piece
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SW; ++s) {
            mbar_init(wfull0 + 8 * s, 1);
            mbar_init(wempty0 + 8 * s, 1);
        }
        for (int s = 0; s < SX; ++s) {
            mbar_init(xfull0 + 8 * s, 1);
            mbar_init(xempty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, kEpiWarps);
        }
        mbar_init(done, 1);
        mbar_init(ring_free, kEpiWarps);
        mbar_init(rx_full, 1);  // armed per group with the bytes the peers will store
        for (int r = 0; r < kMaxCluster; ++r)
            mbar_init(peer_free0 + 8 * r, 1);
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
    cluster_sync();  // every CTA of the cluster has set up its barriers
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- weight producer ----------------
        if (lane == 0) {
            prefetch_tmap(&tmW);
            const uint64_t pol = policy_evict_first();
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            int gi = 0;
            for (int64_t t = cl; t < T && ok; t += CL, ++gi) {
                // The rings hold the peers' partials of the previous group until
                // the epilogue is done with them.
                if (gi > 0 && !mbar_wait(ring_free, (uint32_t)((gi - 1) & 1), limit_ns)) {
                    record_status(status, DEP_DEV_TIMEOUT_PRODUCER);
                    *abort_flag = 1;
                    break;
                }
                for (int kt = kt0; kt < kt1; ++kt) {
                    if (*abort_flag || !mbar_wait(wempty0 + 8 * s, ph ^ 1u, limit_ns)) {
                        if (!*abort_flag)
                            record_status(status, DEP_DEV_TIMEOUT_PRODUCER);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(wfull0 + 8 * s, (uint32_t)S::W_STAGE);
                    for (int g = 0; g < S::TILES; ++g)
                        tma_load_2d(base + (uint32_t)(s * S::W_STAGE + g * kWBytes), S::tile_rows(g) == kBM ? &tmW : &tmW64,
                                    kt * kBK, (int)(t * S::ROWS) + g * kBM, wfull0 + 8 * s, pol);
                    ++issued;
                    if (++s == SW) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // drain: the copies still in flight land before the CTA may leave
            const int64_t n = issued < SW ? issued : SW;
            for (int64_t i = 0; i < n; ++i) {
                if (--s < 0) {
                    s = SW - 1;
                    ph ^= 1u;
                }
                if (!mbar_wait(wfull0 + 8 * s, ph, limit_ns))
                    record_status(status, DEP_DEV_TIMEOUT_PRODUCER);
            }
        }
    } else if (warp == kXWarp) {
        // ---------------- x producer ----------------
        if (lane == 0) {
            prefetch_tmap(&tmX);
            const uint64_t pol = policy_evict_last();
            griddep_wait();  // x may be written by the preceding grid
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            int gi = 0;
            for (int64_t t = cl; t < T && ok; t += CL, ++gi) {
                if (gi > 0 && !mbar_wait(ring_free, (uint32_t)((gi - 1) & 1), limit_ns)) {
                    record_status(status, DEP_DEV_TIMEOUT_PRODUCER);
                    *abort_flag = 1;
                    break;
                }
                for (int kt = kt0; kt < kt1; ++kt) {
                    if (*abort_flag || !mbar_wait(xempty0 + 8 * s, ph ^ 1u, limit_ns)) {
                        if (!*abort_flag)
                            record_status(status, DEP_DEV_TIMEOUT_PRODUCER);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(xfull0 + 8 * s, (uint32_t)S::X_STAGE);
                    tma_load_2d(xbase + (uint32_t)(s * S::X_STAGE), &tmX, kt * kBK, 0, xfull0 + 8 * s, pol);
                    ++issued;
                    if (++s == SX) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            const int64_t n = issued < SX ? issued : SX;
            for (int64_t i = 0; i < n; ++i) {
                if (--s < 0) {
                    s = SX - 1;
                    ph ^= 1u;
                }
                if (!mbar_wait(xfull0 + 8 * s, ph, limit_ns))
                    record_status(status, DEP_DEV_TIMEOUT_PRODUCER);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, NT), idesc64 = tc::idesc_bf16_f32(64, NT);
            int sw = 0, sx = 0, buf = 0;
            uint32_t phw = 0, phx = 0, acce_ph = 0;
            bool ok = true;
            for (int64_t t = cl; t < T && ok; t += CL) {
                if (!mbar_wait(acce0 + 8 * buf, ((acce_ph >> buf) & 1u) ^ 1u, limit_ns)) {
                    record_status(status, DEP_DEV_TIMEOUT_MMA);
                    *abort_flag = 1;
                    break;
                }
                acce_ph ^= 1u << buf;
                tc::fence_after();
                const uint32_t d = tmem + (uint32_t)(buf * S::ACC);
                for (int kt = kt0; kt < kt1; ++kt) {
                    if (*abort_flag || !mbar_wait(wfull0 + 8 * sw, phw, limit_ns) ||
                        !mbar_wait(xfull0 + 8 * sx, phx, limit_ns)) {
                        if (!*abort_flag)
                            record_status(status, DEP_DEV_TIMEOUT_MMA);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const uint32_t wa = base + (uint32_t)(sw * S::W_STAGE);
                    const uint64_t bd = tc::desc_sw128(xbase + (uint32_t)(sx * S::X_STAGE));
#pragma unroll
                    for (int j = 0; j < kBK / kUmmaK; ++j) {
                        // advance along K inside the 128-byte swizzle row: 32 bytes per step
                        const uint64_t off = (uint64_t)((j * kUmmaK * 2) >> 4);
                        const uint32_t acc = (kt != kt0 || j > 0) ? 1u : 0u;
#pragma unroll
                        for (int g = 0; g < S::TILES; ++g)
                            tc::mma_bf16(d + (uint32_t)(g * NT), tc::desc_sw128(wa + (uint32_t)(g * kWBytes)) + off,
                                         bd + off, S::tile_rows(g) == kBM ? idesc : idesc64, acc);
                    }
                    tc::commit(wempty0 + 8 * sw);  // the stages are free once these MMAs finish
                    tc::commit(xempty0 + 8 * sx);
                    if (++sw == SW) {
                        sw = 0;
                        phw ^= 1u;
                    }
                    if (++sx == SX) {
                        sx = 0;
                        phx ^= 1u;
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
        griddep_wait();  // y may still be in use by the preceding grid
        const int e = warp - 2;         // chunk index within a piece
        const int q = warp & 3;         // TMEM lane quadrant this warp may access
        const int h = e >> 2;           // accumulator column half
        const int ms = max_share(S::NCB, k);
        // Column block cb of this warp: accumulator columns h HALF + cb CBW ..,
        // tile col / NT, batch rows from col % NT.
        auto col_tile = [&](int cb) { return (h * S::HALF + cb * S::CBW) / NT; };
        auto col_b0 = [&](int cb) { return (h * S::HALF + cb * S::CBW) % NT; };
        // The weight row of this lane in tile g, and whether the lane holds one: a
        // 128-row tile has row 32 q + lane in TMEM lane quadrant q; the 64-row
        // (M = 64) tile has rows 16 q .. 16 q + 15 in lanes 0-15 of quadrant q.
        auto tile_row = [&](int g) { return S::tile_rows(g) == kBM ? 32 * q + lane : 16 * q + lane; };
        auto lane_has_row = [&](int g) { return S::tile_rows(g) == kBM || lane < 16; };
        // Where sender `from` puts column block cb (of a share starting at cb0)
        // in the receiving CTA: [sender slot][warp][block of the share][lane][CBW].
        auto recv_off = [&](int from, int to, int cb, int cb0) -> uint32_t {
            const int js = from - (from > to ? 1 : 0);
            return (uint32_t)(((js * kEpiWarps + e) * ms + (cb - cb0)) * S::CB_BYTES);
        };
        uint32_t accf_ph = 0;
        int buf = 0, gi = 0;
        bool ok = true;
        const bool elected = warp == 2 && lane == 0;  // issues the y stores
        const uint32_t stg = base + (uint32_t)stage_offset(S::NCB, k, S::CB_BYTES);
        int stg_i = 0;  // y staging buffers used so far
        for (int64_t t = cl; t < T; t += CL, ++gi) {
            bool got = ok && mbar_wait(accf0 + 8 * buf, (accf_ph >> buf) & 1u, limit_ns);
            if (ok && !got)
                record_status(status, DEP_DEV_TIMEOUT_EPILOGUE);
            ok = epi_all(got);  // every epilogue warp takes the same path from here
            if (!ok) {
                *abort_flag = 1;
                break;
            }
            accf_ph ^= 1u << buf;
            tc::fence_after();
            const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * S::ACC + h * S::HALF);
            const uint32_t par = (uint32_t)(gi & 1);
            if (k > 1) {
                // 1. This CTA's MMAs of the group are done: its rings are idle.  Arm
                //    the receive barrier with the bytes the peers will store, then
                //    tell them.
                if (warp == 2) {
                    if (lane == 0) {
                        uint32_t nb = 0;
                        for (int cb = share_begin(rank, S::NCB, k); cb < share_begin(rank + 1, S::NCB, k); ++cb)
                            nb += col_b0(cb) < B ? (uint32_t)(S::CB_ROWS * S::CBW * 4) : 0u;
                        mbar_arrive_expect_tx(rx_full, nb * (uint32_t)(k - 1));
                    }
                    __syncwarp();
                    if (lane < k && lane != rank)
                        mbar_arrive_peer(peer_addr(peer_free0 + 8 * rank, (uint32_t)lane));
                }
                // 2. Each peer's share of this warp's columns into the peer's rings.
                for (int p = 0; p < k; ++p) {
                    if (p == rank)
                        continue;
                    if (!mbar_wait_cluster(peer_free0 + 8 * p, par, limit_ns)) {
                        record_status(status, DEP_DEV_TIMEOUT_EPILOGUE);
                        ok = false;
                    }
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok)
                        break;
                    const int c0 = share_begin(p, S::NCB, k), c1 = share_begin(p + 1, S::NCB, k);
                    const uint32_t pbar = peer_addr(rx_full, (uint32_t)p);
                    for (int cb = c0; cb < c1; ++cb) {
                        if (col_b0(cb) >= B || !dbg_range(recv_off(rank, p, cb, c0), S::CB_BYTES, (unsigned)RING, status))
                            continue;
                        const uint32_t dst = peer_addr(base + recv_off(rank, p, cb, c0), (uint32_t)p);
                        const bool has = lane_has_row(col_tile(cb));  // lanes without a row send nothing
#pragma unroll 1
                        for (int c16 = 0; c16 < S::CBW; c16 += 16) {
                            __syncwarp();  // tcgen05.ld is warp-collective: every lane, converged
                            uint32_t v[16];
                            tc::ld16(tq + (uint32_t)(cb * S::CBW + c16), v);
                            tc::wait_ld();
                            if (has) {
#pragma unroll
                                for (int i = 0; i < 4; ++i)
                                    st_async_peer_v4(dst + (uint32_t)(((c16 / 4 + i) * 32 + lane) * 16),
                                                     __uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                                     __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]),
                                                     pbar);
                            }
                        }
                    }
                }
                // 3. Every peer's part of this CTA's share has landed.
                if (ok && !mbar_wait_cluster(rx_full, par, limit_ns)) {
                    record_status(status, DEP_DEV_TIMEOUT_EPILOGUE);
                    ok = false;
                }
                ok = epi_all(ok);
            }
            // 4. This CTA's share: the K pieces in rank order, its own from TMEM.
            const int c0 = k > 1 ? share_begin(rank, S::NCB, k) : 0;
            const int c1 = k > 1 ? share_begin(rank + 1, S::NCB, k) : S::NCB;
            for (int cb = c0; cb < c1 && ok; ++cb) {
                const int b0 = col_b0(cb);  // the same for every epilogue warp
                if (b0 >= B)
                    continue;
                const int g = col_tile(cb);
                const bool has = lane_has_row(g);
                const int rt = tile_row(g), pitch = S::tile_rows(g);
                const int64_t n = t * S::ROWS + (int64_t)g * kBM + rt;
                // y staging buffer of this column block: [h][batch row j][tile rows]
                uint16_t *sy = reinterpret_cast<uint16_t *>(smem + (stg - base) +
                                                            (size_t)(stg_i & 1) * (stage_bytes(S::CBW) / 2));
                if (use_tma_y) {
                    if (elected)
                        bulk_wait_read1();  // the store issued from this buffer two blocks ago has read it
                    epi_sync();
                }
#pragma unroll 1
                for (int c16 = 0; c16 < S::CBW; c16 += 16) {
                    __syncwarp();
                    uint32_t own[16];
                    tc::ld16(tq + (uint32_t)(cb * S::CBW + c16), own);
                    tc::wait_ld();
                    float sum[16];
#pragma unroll 1
                    for (int p = 0; p < k; ++p) {
                        float v[16];
                        if (p == rank) {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                v[j] = __uint_as_float(own[j]);
                        } else if (dbg_range(recv_off(p, rank, cb, c0), S::CB_BYTES, (unsigned)RING, status)) {
                            const float4 *src = reinterpret_cast<const float4 *>(
                                smem + recv_off(p, rank, cb, c0) + (size_t)c16 * 128);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const float4 f = src[i * 32 + lane];
                                v[4 * i] = f.x;
                                v[4 * i + 1] = f.y;
                                v[4 * i + 2] = f.z;
                                v[4 * i + 3] = f.w;
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                v[j] = 0.0f;  // (bounds-checked builds only: the check above failed)
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            sum[j] = p == 0 ? v[j] : sum[j] + v[j];
                    }
                    if (use_tma_y) {
                        if (has) {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                sy[(size_t)h * S::CBW * kBM + (size_t)(c16 + j) * pitch + rt] = to_bf16(sum[j]);
                        }
                    } else if (has) {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (b0 + c16 + j < B && n < N && dbg_ok((int64_t)(b0 + c16 + j) * N + n, bd.y, status))
                                y[(int64_t)(b0 + c16 + j) * N + n] = to_bf16(sum[j]);
                    }
                }
                if (use_tma_y) {
                    fence_proxy_async_smem();
                    epi_sync();
                    if (elected) {
                        // two boxes [CBW batch rows x tile rows], one per column half;
                        // rows past N and batch rows past B are clipped by the store
                        for (int hh = 0; hh < 2; ++hh) {
                            const int gg = (hh * S::HALF + cb * S::CBW) / NT;
                            tma_store_2d(S::tile_rows(gg) == kBM ? &tmY : &tmY64,
                                         smem_u32(sy) + (uint32_t)(hh * S::CBW * kBM * 2), (int)(t * S::ROWS) + gg * kBM,
                                         b0);
                        }
                        bulk_commit();
                    }
                    ++stg_i;
                }
            }
            if (use_tma_y) {
                if (elected)
                    bulk_wait_read0();  // the staging area (part of the rings) is read out
                epi_sync();
            }
            // 5. The rings and the accumulator are free again.
            tc::fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(ring_free);
                mbar_arrive(acce0 + 8 * buf);
            }
            if (S::BUFS == 2)
                buf ^= 1;
        }
    }

    if (warp == 2 && lane == 0)
        bulk_wait0();  // the y stores are complete
    __syncwarp();
    tc::fence_before();
    __syncthreads();
    cluster_sync();  // no CTA leaves while a peer may still write into its shared memory
    if (warp == 1) {
        tc::fence_after();
        tc::dealloc(tmem, S::TMEM_COLS);
    }
}

}  // namespace
}  // namespace dep

namespace dep {
namespace {

constexpr size_t kBudget = (size_t)kMaxDynamicSmem;

// x stages that fit beside `sw` weight stages (0 if fewer than two).
int x_stages(int sw, int w_stage, int x_stage)
{
    for (int sx = kMaxXStages; sx >= 2; --sx) {
        const size_t need = 1024 + (size_t)sw * w_stage + (size_t)sx * x_stage + (size_t)barrier_count(sw, sx) * 8 + 16;
        if (need <= kBudget)
            return sx;
    }
    return 0;
}

// Shared memory of a launch; at least half of an SM's, so that a CTA never
// shares its SM (and TMEM) with another CTA of this kernel.
size_t cluster_smem(int sw, int sx, int w_stage, int x_stage)
{
    const size_t need = 1024 + (size_t)sw * w_stage + (size_t)sx * x_stage + (size_t)barrier_count(sw, sx) * 8 + 16;
    const size_t floor_b = (size_t)kMaxDynamicSmem / 2 + 1024;
    return need > floor_b ? need : floor_b;
}

template <int NT, int G>
bool valid_shape(const dep_tactic_t &t)
{
    using S = ClusterShape<NT, G>;
    const int sx = x_stages(t.stages, S::W_STAGE, S::X_STAGE);
    if (!sx)
        return false;
    const size_t ring = (size_t)t.stages * S::W_STAGE + (size_t)sx * S::X_STAGE;
    // the peers' partials and the y staging fit in the idle rings
    return stage_offset(S::NCB, t.splits, S::CB_BYTES) + stage_bytes(S::CBW) <= ring;
}

template <int NT, int G>
cudaError_t prepare()
{
    static std::atomic<uint64_t> devices{0};
    return set_smem_attr(tc_cluster_kernel<NT, G>, devices);
}

template <int NT, int G>
cudaError_t run_shape(const dep_tactic_t &t, const RunArgs &a)
{
    using S = ClusterShape<NT, G>;
    cudaError_t e = prepare<NT, G>();
    if (e != cudaSuccess)
        return e;
    CUtensorMap tmW, tmW64, tmX, tmY, tmY64;
    if (encode_bf16_2d(&tmW, a.W, (uint64_t)a.K, (uint64_t)a.N, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B) !=
            CUDA_SUCCESS ||
        encode_bf16_2d(&tmW64, a.W, (uint64_t)a.K, (uint64_t)a.N, kBK, 64, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // y goes out in bulk tensor stores when its rows are 16-byte multiples (a
    // tensor map's row pitch must be), else by plain stores.
    const bool tma_y = a.N % 8 == 0;
    const int64_t T = (a.N + S::ROWS - 1) / S::ROWS, KT = (a.K + kBK - 1) / kBK;
    const int k = (int)(t.splits < KT ? t.splits : KT);  // every rank gets at least one k-tile
    int64_t clusters = t.ctas / t.splits;
    clusters = clusters < 1 ? 1 : (clusters > T ? T : clusters);
    const int sx = x_stages(t.stages, S::W_STAGE, S::X_STAGE);
    const size_t smem = cluster_smem(t.stages, sx, S::W_STAGE, S::X_STAGE);
    for (int32_t r0 = 0; r0 < a.B; r0 += NT) {
        const int32_t rows = a.B - r0 < NT ? a.B - r0 : NT;
        if (encode_bf16_2d(&tmX, a.x + (size_t)r0 * a.K, (uint64_t)a.K, (uint64_t)rows, kBK, NT,
                           CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        if (tma_y) {
            if (encode_bf16_2d(&tmY, a.y + (size_t)r0 * a.N, (uint64_t)a.N, (uint64_t)rows, kBM, S::CBW,
                               CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS ||
                encode_bf16_2d(&tmY64, a.y + (size_t)r0 * a.N, (uint64_t)a.N, (uint64_t)rows, 64, S::CBW,
                               CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
                return cudaErrorInvalidValue;
        } else {
            tmY = tmY64 = tmX;  // not used
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(clusters * k));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = a.stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)k;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = a.pdl ? 1 : 0;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        e = cudaLaunchKernelEx(&cfg, tc_cluster_kernel<NT, G>, tmW, tmW64, tmX, tmY, tmY64, a.y + (size_t)r0 * a.N,
                               (int)rows,
                               (int)a.N, (int)a.K, (int)t.stages, sx, tma_y ? 1 : 0, a.status, a.bounds(rows, smem),
                               a.wait_limit_ns);
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

template <int NT, int G>
cudaError_t prepare_shape(const dep_tactic_t &)
{
    return prepare<NT, G>();
}

// The instantiation of a tactic: MMA width (cols) x group (tile_n = 256, 192 or
// 512 weight rows: G = 2, 3 (a 128-row and a 64-row tile) or 4).
#define DEP_CLUSTER_DISPATCH(NAME, RET, FN, BAD)                                             \
    RET NAME(const dep_tactic_t &t)                                                          \
    {                                                                                        \
        const int g = t.tile_n == 192 ? 3 : t.tile_n / kBM;                                  \
        switch (t.cols) {                                                                    \
        case 32: return g == 4 ? FN<32, 4>(t) : g == 2 ? FN<32, 2>(t) : BAD;                 \
        case 64: return g == 4 ? FN<64, 4>(t) : g == 3 ? FN<64, 3>(t) : g == 2 ? FN<64, 2>(t) : BAD;     \
        case 128: return g == 4 ? FN<128, 4>(t) : g == 3 ? FN<128, 3>(t) : g == 2 ? FN<128, 2>(t) : BAD; \
        case 256: return g == 3 ? FN<256, 3>(t) : g == 2 ? FN<256, 2>(t) : BAD;             \
        default: return BAD;                                                                 \
        }                                                                                    \
    }

DEP_CLUSTER_DISPATCH(valid_for, bool, valid_shape, false)
DEP_CLUSTER_DISPATCH(prepare_for, cudaError_t, prepare_shape, cudaErrorInvalidValue)
#undef DEP_CLUSTER_DISPATCH

}  // namespace

bool cluster_valid(const dep_tactic_t &t)
{
    if (t.kind != DEP_KIND_TC_CLUSTER || t.tile_k != kBK ||
        (t.tile_n != 2 * kBM && t.tile_n != 4 * kBM && t.tile_n != 192))
        return false;
    if (t.splits < 1 || t.splits > kMaxCluster || t.ctas < t.splits || t.ctas % t.splits)
        return false;  // whole clusters of 1..8 CTAs
    if (t.stages < 2 || t.stages > 16)
        return false;
    return valid_for(t);
}

cudaError_t cluster_prepare_device()
{
    for (int32_t cols : {32, 64, 128, 256})
        for (int32_t rows : {256, 192, 512}) {
            if (cols * (rows == 192 ? 2 : rows / kBM) > 512 || (rows == 192 && cols == 32))
                continue;
            dep_tactic_t t{};
            t.cols = cols;
            t.tile_n = rows;
            const cudaError_t e = prepare_for(t);
            if (e != cudaSuccess)
                return e;
        }
    return cudaSuccess;
}

cudaError_t cluster_run(const dep_tactic_t &t, const RunArgs &a)
{
    const int g = t.tile_n == 192 ? 3 : t.tile_n / kBM;
    switch (t.cols) {
    case 32: return g == 4 ? run_shape<32, 4>(t, a) : run_shape<32, 2>(t, a);
    case 64: return g == 4 ? run_shape<64, 4>(t, a) : g == 3 ? run_shape<64, 3>(t, a) : run_shape<64, 2>(t, a);
    case 128: return g == 4 ? run_shape<128, 4>(t, a) : g == 3 ? run_shape<128, 3>(t, a) : run_shape<128, 2>(t, a);
    case 256: return g == 3 ? run_shape<256, 3>(t, a) : run_shape<256, 2>(t, a);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace dep
