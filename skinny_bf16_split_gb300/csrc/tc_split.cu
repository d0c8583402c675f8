// tc_split.cu -- tcgen05 tactic with a fixed K split and dynamic scheduling.
//
// Computes y[B,N] = BF16(x[B,K] . W[N,K]^T), BF16 products accumulated in FP32
// (runtime.hybrid page, HybridAttention.__init__: past the split-K rows the
// projection runs the stock FP32-accumulated BF16 GEMM; runtime.dep page,
// DepProjection), like the stream-K tensor-core tactic, with another schedule:
//
//  * Each 128-row weight tile is cut into S fixed pieces along K (piece p
//    covers k-tiles [p KT / S, (p+1) KT / S)).  A work item is one (tile,
//    piece) pair; item i is tile i / S, piece i % S.
//  * Blocks take items dynamically: item blockIdx.x first, then the next free
//    item from an integer counter, so a block that streams faster takes more
//    items and the blocks finish together (a static split ends when its
//    slowest block does).  The last block to finish taking items resets the
//    counter for the next launch.
//  * Swap-AB MMAs as in the stream-K kernel: M = BM = 128 (or 64) weight rows,
//    N = the batch padded to NT, K = 16 per instruction; 128-byte-swizzled TMA
//    stages of tile_k / 64 slices; accumulators in TMEM, two buffers.  The first
//    stages are issued by thread 0 right after the barrier set-up, while warp 1
//    allocates TMEM.
//  * 64-row tiles at NT <= 32 take slices in pairs when a stage has an even
//    number of them: an M = 64 MMA costs as long as an M = 128 one, so one
//    M = 128, N = 2 NT instruction reads slice 2j as A rows 0-63 and slice 2j+1
//    (the next 8 KB) as rows 64-127, against x slices 2j and 2j+1 as B rows
//    0..NT-1 and NT..2NT-1.  Lanes 0-63 / columns [0, NT) of D collect the even
//    slices, lanes 64-127 / columns [NT, 2 NT) the odd ones (the two other
//    blocks of D are never read).  The epilogue warps of lane quadrants 2-3
//    hand their sums to those of quadrants 0-1 through shared memory, and a
//    row's partial is (even slices) + (odd slices), each issuer 0's plus issuer
//    1's, in FP32: half the instructions per weight byte, same determinism.
//  * One thread issues a tcgen05.mma about every 67 cycles whatever its M and
//    N (up to N = 128), which at N <= 64 is less work per instruction than the
//    tensor pipe can do: a block with one issuer consumes about 60 weight bytes
//    per cycle, barely ahead of its share of HBM, and drains a prefetched ring
//    slowly.  For NT <= 32 two warps issue: each takes a fixed half of every
//    stage's 16-column K steps into its own accumulator, and the epilogue adds
//    the two in issuer order (FP32), so the result stays deterministic.
//  * Pieces are exchanged through the plan's exchange region, one 64-bit word
//    per (tile, piece, b, row): the FP32 partial in the low half and a "full"
//    flag in the high half, written by one single-copy-atomic store (no fence,
//    no atomic counter).  The block that runs the last piece of a tile reduces:
//    it waits (bounded) until the words of pieces 0..S-2 are full, adds them in
//    piece order and its own piece last, rounds to BF16, and clears the flags
//    for the next launch (the values stay for inspection).  Which block ran
//    which piece does not enter the arithmetic, so results are identical from
//    run to run and equal to BF16 of the ordered FP32 sum of the pieces.  With
//    S = 1 a tile is one item and y is stored directly.
//    No deadlock: items are handed out in increasing order and the pieces of a
//    tile precede its last piece, so every piece a reducer waits for is already
//    held by a running block (or was run earlier by the same block), and the
//    earliest pending reduction never waits on a later one.
//  * Warp roles: warp 0 TMA producer (takes the items), warp 1 TMEM owner and
//    MMA issuer 0, warp 2 MMA issuer 1 (NT <= 32), warps 3-6 epilogue.  The
//    producer tags each stage with its item and first/last flags; issuer 0
//    passes the item of each finished accumulator to the epilogue through a tag
//    slot and its own mbarrier.
//  * Every wait is bounded in time; on a give-up the block records a code, lets
//    every role finish, waits for its MMAs and copies, and frees TMEM.
#include <cuda_bf16.h>

#include "exchange.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace dep {
namespace {

constexpr int kBK = 64;       // columns per slice: one 128-byte swizzle row
constexpr int kUmmaK = 16;    // K of one kind::f16 MMA
constexpr int kThreads = 224; // warp 0 TMA, warps 1-2 MMA (warp 1 owns TMEM), warps 3-6 epilogue
constexpr int kEpiWarps = 4;
constexpr int kMaxSplits = 64;

// BM = weight rows per tile = MMA M (64 or 128); NT = MMA N (the padded batch).
template <int NT, int BM>
struct SplitShape {
    static constexpr int A_BYTES = BM * kBK * 2;  // one weight slice: 8 or 16 KB
    static constexpr int B_BYTES = NT * kBK * 2;
    static constexpr int ATOM = A_BYTES + B_BYTES;
    // MMA issuers, each with its own accumulator per buffer: two at N <= 32,
    // the same rule as the stream-K kernel, whose results these must equal.
    static constexpr int ISSUERS = NT <= 32 ? 2 : 1;
    // 64-row tiles at N <= 32 issue slice pairs (when a stage has an even number
    // of slices): one M = 128, N = 2 NT instruction covers two slices, the even
    // one in TMEM lanes 0-63 / columns [0, NT), the odd one in lanes 64-127 /
    // columns [NT, 2 NT).  An M = 64 instruction takes as long as an M = 128
    // one, so this halves the instructions per weight byte.
    static constexpr bool PAIRABLE = BM == 64 && NT <= 32;
    static constexpr int ACC_MAX = PAIRABLE ? 2 * NT : NT;  // accumulator columns
    static constexpr uint32_t TMEM_COLS = 2 * ISSUERS * ACC_MAX < 32 ? 32 : 2 * ISSUERS * ACC_MAX;
    // The odd slices' sums pass from the warps reading TMEM lanes 64-127 to the
    // warps owning the rows: [buffer][lane quadrant pair][column][lane] floats.
    static constexpr int XFER_BYTES = PAIRABLE ? 2 * 2 * NT * 32 * 4 : 0;
};

// Shared memory after the 1 KB-aligned ring: the slice-pair hand-off area;
// full[stages], empty[stages], accf[2], acce[2], tagb[2], done, hand[2][2];
// then the stage tags, the accumulator items, the TMEM address and the abort flag.
__host__ __device__ inline size_t split_smem_bytes(int stages, int stage_bytes, int xfer_bytes)
{
    return 1024 + (size_t)stages * stage_bytes + (size_t)xfer_bytes + (size_t)(2 * stages + 11) * 8 +
           (size_t)stages * 8 + 16;
}

__device__ __forceinline__ int piece_begin(int p, int KT, int S)
{
    return (int)(((int64_t)p * KT) / S);
}

__device__ __forceinline__ uint16_t to_bf16(float v)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}


template <int NT, int BM>
__global__ void __launch_bounds__(kThreads, 1)
    tc_split_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                    uint16_t *__restrict__ y, int B, int N, int K, int stages, int atoms, int S, int tma3,
                    unsigned long long *__restrict__ xch, int *__restrict__ dispenser,
                    int *__restrict__ status, const Bounds bd, uint64_t limit_ns)
{
    using Sh = SplitShape<NT, BM>;
    const int STAGE = atoms * Sh::ATOM;
    const int KG = atoms * kBK;  // columns per k-tile (one stage)
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle tiles need 1 KB alignment
    uint8_t *smem = smem_raw + (base - raw);
    if (!dbg_ok((base - raw) + split_smem_bytes(stages, STAGE, Sh::XFER_BYTES) - 1024 - 1, bd.smem, status))
        return;  // the ring, barriers, tags and TMEM slot must lie in the launch's shared memory
    float *xfer = reinterpret_cast<float *>(smem + (size_t)stages * STAGE);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)stages * STAGE + Sh::XFER_BYTES);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = full0 + 8 * stages;
    const uint32_t accf0 = empty0 + 8 * stages;  // accumulator final, 2 buffers
    const uint32_t acce0 = accf0 + 16;           // accumulator drained, 2 buffers
    const uint32_t tagb0 = acce0 + 16;           // accumulator's item published, 2 buffers
    const uint32_t done = tagb0 + 16;            // all MMAs complete
    const uint32_t hand0 = done + 8;             // odd-slice sums handed over, [buffer][quadrant pair]
    int2 *tags = reinterpret_cast<int2 *>(bars + 2 * stages + 11);  // (item, flags); item < 0: end
    volatile int *acc_item = reinterpret_cast<volatile int *>(tags + stages);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tags + stages) + 2;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int T = (N + BM - 1) / BM, KT = (K + KG - 1) / KG, I = T * S;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool pair = Sh::PAIRABLE && (atoms & 1) == 0;  // slice-pair MMAs
    const int ACC = pair ? 2 * NT : NT;                   // columns of one accumulator
    int *grab = dispenser, *finished = dispenser + 1;

    // Producer state; the producer is thread 0 (warp 0, lane 0).
    uint64_t pol_w = 0, pol_x = 0;
    int item = blockIdx.x;  // the grid never exceeds the item count
    int tile = item / S, kt = piece_begin(item % S, KT, S), kt_end = piece_begin(item % S + 1, KT, S);
    const int kt0 = kt;
    const int pre = (kt_end - kt) < stages ? (kt_end - kt) : stages;
    auto stage_addr = [&](int st) { return base + (uint32_t)(st * STAGE); };
    auto issue_w = [&](int st) {
        const int flags = (kt == piece_begin(item % S, KT, S) ? 1 : 0) | (kt == kt_end - 1 ? 2 : 0);
        tags[st] = make_int2(item, flags);
        mbar_arrive_expect_tx(full0 + 8 * st, (uint32_t)STAGE);
        if (tma3)  // the stage's slices in one copy (column-block view of W)
            tma_load_3d(stage_addr(st), &tmW, 0, tile * BM, kt * atoms, full0 + 8 * st, pol_w);
        else
            for (int a = 0; a < atoms; ++a)
                tma_load_2d(stage_addr(st) + (uint32_t)(a * Sh::A_BYTES), &tmW, kt * KG + a * kBK, tile * BM,
                            full0 + 8 * st, pol_w);
    };
    auto issue_x = [&](int st, int k_tile) {
        const uint32_t xs = stage_addr(st) + (uint32_t)(atoms * Sh::A_BYTES);
        if (tma3)
            tma_load_3d(xs, &tmX, 0, 0, k_tile * atoms, full0 + 8 * st, pol_x);
        else
            for (int a = 0; a < atoms; ++a)
                tma_load_2d(xs + (uint32_t)(a * Sh::B_BYTES), &tmX, k_tile * KG + a * kBK, 0, full0 + 8 * st,
                            pol_x);
    };

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmX);
        for (int s = 0; s < stages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, Sh::ISSUERS);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, Sh::ISSUERS);
            mbar_init(acce0 + 8 * b, kEpiWarps);
            mbar_init(tagb0 + 8 * b, 1);
        }
        mbar_init(done, Sh::ISSUERS);
        for (int h = 0; h < 4; ++h)
            mbar_init(hand0 + 8 * h, 32);
        *abort_flag = 0;
        fence_mbar_init();
        griddep_launch_dependents();
        // Phase 1, while warp 1 allocates TMEM: the weight is not written by
        // preceding work -- fill the ring with the first k-tiles of the first item.
        pol_w = policy_evict_first();
        pol_x = policy_evict_last();
        for (int i = 0; i < pre; ++i, ++kt)
            issue_w(i);
    }
    if (warp == 1) {
        tc::alloc(smem_u32(tmem_slot), Sh::TMEM_COLS);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer: takes the items ----------------
        if (lane == 0) {
            // Phase 2: after the preceding grid -- x of the filled stages, then the
            // rest of the items (taken from the counter).
            griddep_wait();
            for (int i = 0; i < pre; ++i)
                issue_x(i, kt0 + i);
            int s = pre % stages;
            uint32_t ph = pre == stages ? 1u : 0u;
            int64_t issued = pre;
            bool ok = true;
            for (;;) {
                if (kt == kt_end) {  // the item is fully issued: take the next one
                    item = (int)gridDim.x + atomicAdd(grab, 1);
                    if (item < I) {
                        tile = item / S;
                        kt = piece_begin(item % S, KT, S);
                        kt_end = piece_begin(item % S + 1, KT, S);
                    }
                }
                if (*abort_flag) {
                    ok = false;
                    break;
                }
                if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, limit_ns)) {
                    record_status(status, DEP_DEV_TIMEOUT_PRODUCER);
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                if (item >= I) {  // end of the stream: an empty stage tagged -1
                    tags[s] = make_int2(-1, 0);
                    mbar_arrive(full0 + 8 * s);
                    break;
                }
                issue_w(s);
                issue_x(s, kt);
                ++kt;
                ++issued;
                if (++s == stages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            // Drain: walk back over the most recent fills from stage s.  After an
            // end marker stage s holds the marker, so at most stages - 1 copies can
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
            // The last block to finish taking items resets the counter.
            if (atomicAdd(finished, 1) == (int)gridDim.x - 1) {
                *grab = 0;
                *finished = 0;
            }
        }
    } else if (warp == 1 || warp == 2) {
        // ---------------- MMA issuers ----------------
        // Issuer mi takes K steps [mi H, (mi + 1) H) of every stage (H = the
        // stage's steps / issuers) into its own accumulator of each buffer.
        const int mi = warp - 1;
        if (lane == 0 && mi < Sh::ISSUERS) {
            constexpr uint32_t idesc1 = tc::idesc_bf16_f32(BM, NT);
            constexpr uint32_t idesc2 = Sh::PAIRABLE ? tc::idesc_bf16_f32(128, 2 * NT) : idesc1;
            const uint32_t idesc = pair ? idesc2 : idesc1;
            // K steps of a stage: 4 per slice, or per slice pair
            const int H = (pair ? atoms / 2 : atoms) * (kBK / kUmmaK) / Sh::ISSUERS;
            int s = 0, buf = 0;
            uint32_t ph = 0, acce_ph = 0;
            uint32_t accumulate = 0;
            for (;;) {
                if (!mbar_wait(full0 + 8 * s, ph, limit_ns)) {
                    record_status(status, DEP_DEV_TIMEOUT_MMA);
                    *abort_flag = 1;
                    break;
                }
                tc::fence_after();
                const int2 tag = tags[s];
                if (tag.x < 0 || (tag.y & 1)) {
                    // A new item (or the end): take accumulator buffer `buf` once the
                    // epilogue has drained its previous use.
                    if (!mbar_wait(acce0 + 8 * buf, ((acce_ph >> buf) & 1u) ^ 1u, limit_ns)) {
                        record_status(status, DEP_DEV_TIMEOUT_MMA);
                        *abort_flag = 1;
                        break;
                    }
                    acce_ph ^= 1u << buf;
                    tc::fence_after();
                    accumulate = 0;
                }
                if (tag.x < 0) {  // issuer 0 hands the end marker to the epilogue
                    if (mi == 0) {
                        acc_item[buf] = -1;
                        mbar_arrive(tagb0 + 8 * buf);
                    }
                    break;
                }
                const uint32_t d = tmem + (uint32_t)((buf * Sh::ISSUERS + mi) * ACC);
                const uint32_t st = base + (uint32_t)(s * STAGE);
                if (pair)  // step i: slices 2 (i / 4) and 2 (i / 4) + 1 at K offset 16 (i % 4)
                    tc::mma_stage<2 * Sh::A_BYTES, 2 * Sh::B_BYTES>(d, st, st + (uint32_t)(atoms * Sh::A_BYTES), mi * H,
                                                                    H, idesc, accumulate);
                else
                    tc::mma_stage<Sh::A_BYTES, Sh::B_BYTES>(d, st, st + (uint32_t)(atoms * Sh::A_BYTES), mi * H, H,
                                                            idesc, accumulate);
                tc::commit(empty0 + 8 * s);  // the stage is free once both issuers' MMAs finish
                if (++s == stages) {
                    s = 0;
                    ph ^= 1u;
                }
                if (tag.y & 2) {  // the item's last k-tile: publish the accumulator
                    if (mi == 0)
                        acc_item[buf] = tag.x;
                    tc::commit(accf0 + 8 * buf);  // complete once both issuers' MMAs finish
                    if (mi == 0)
                        mbar_arrive(tagb0 + 8 * buf);
                    buf ^= 1;
                }
            }
            tc::commit(done);  // TMEM is freed at the end: wait for every MMA
            if (!mbar_wait(done, 0, limit_ns))
                record_status(status, DEP_DEV_TIMEOUT_MMA);
        }
    } else {
        // ---------------- epilogue warps ----------------
        griddep_wait();  // the exchange words and y may still be in use by the preceding grid
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        // M = 128: tile row r is TMEM lane r.  M = 64: rows 16q..16q+15 are lanes
        // 0-15 of quadrant q (lanes 16-31 hold nothing of this MMA).  Slice pairs:
        // row r is lane r (even slices) and lane 64 + r (odd slices); quadrants 0-1
        // own the rows, quadrants 2-3 hand their sums to them.
        const bool odd = pair && q >= 2;
        const int row = pair ? 32 * (q & 1) + lane : (BM == 128 ? 32 * q + lane : 16 * q + lane);
        const bool has_row = pair ? !odd : (BM == 128 || lane < 16);
        uint32_t tag_ph = 0, accf_ph = 0, hand_ph = 0;
        int buf = 0;
        for (;;) {
            if (!mbar_wait(tagb0 + 8 * buf, (tag_ph >> buf) & 1u, limit_ns)) {
                record_status(status, DEP_DEV_TIMEOUT_EPILOGUE);
                *abort_flag = 1;
                break;
            }
            tag_ph ^= 1u << buf;
            const int item = acc_item[buf];
            if (item < 0)
                break;
            if (!mbar_wait(accf0 + 8 * buf, (accf_ph >> buf) & 1u, limit_ns)) {
                record_status(status, DEP_DEV_TIMEOUT_EPILOGUE);
                *abort_flag = 1;
                break;
            }
            accf_ph ^= 1u << buf;
            tc::fence_after();
            const int t = item / S, piece = item % S;
            const int64_t n = (int64_t)t * BM + row;
            const bool mine = has_row && n < N;  // this lane's output row exists
            // buffer buf's accumulators: issuer 0's, then issuer 1's (ACC columns each)
            const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * Sh::ISSUERS * ACC);
            float *hand = xfer + (size_t)(2 * buf + (q & 1)) * NT * 32 + lane;  // [column][lane]
            const uint32_t hand_bar = hand0 + 8 * (uint32_t)(2 * buf + (q & 1));
            if (odd) {
                // Columns [NT, 2 NT) of lanes 64-127: the odd slices' sums, issuer
                // 0's plus issuer 1's, handed to the warp that owns these rows.
#pragma unroll 1
                for (int c0 = 0; c0 < NT && c0 < B; c0 += 16) {
                    __syncwarp();
                    uint32_t v[16], v1[16];
                    tc::ld16(taddr + (uint32_t)(NT + c0), v);
                    tc::ld16(taddr + (uint32_t)(ACC + NT + c0), v1);
                    tc::wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        hand[(c0 + j) * 32] = __uint_as_float(v[j]) + __uint_as_float(v1[j]);
                }
                mbar_arrive(hand_bar);
                tc::fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(acce0 + 8 * buf);
                buf ^= 1;
                continue;
            }
            if (pair) {
                if (!mbar_wait(hand_bar, (hand_ph >> buf) & 1u, limit_ns)) {
                    record_status(status, DEP_DEV_TIMEOUT_EPILOGUE);
                    *abort_flag = 1;
                    break;
                }
                hand_ph ^= 1u << buf;
            }
            // tile t's exchange words, [piece][b][row]
            unsigned long long *tile_x = xch + (int64_t)t * S * NT * BM + row;
            bool ok = true;
#pragma unroll 1
            for (int c0 = 0; c0 < NT && c0 < B; c0 += 16) {
                __syncwarp();  // tcgen05.ld is warp-collective: every lane, converged
                uint32_t v[16], v1[16];
                tc::ld16(taddr + (uint32_t)c0, v);
                if (Sh::ISSUERS == 2)
                    tc::ld16(taddr + (uint32_t)(ACC + c0), v1);
                tc::wait_ld();
                if (Sh::ISSUERS == 2) {  // the block's partial: issuer 0's half of K, then issuer 1's
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(v1[j]));
                }
                if (pair) {  // (even slices) + (odd slices), each issuer 0 + issuer 1
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        v[j] = __float_as_uint(__uint_as_float(v[j]) + hand[(c0 + j) * 32]);
                }
                if (S == 1) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < B && mine && dbg_ok((int64_t)(c0 + j) * N + n, bd.y, status))
                            y[(int64_t)(c0 + j) * N + n] = to_bf16(__uint_as_float(v[j]));
                    continue;
                }
                const int64_t tile_w = (int64_t)t * S * NT * BM + row;  // tile t's words start here
                const int64_t own_w = tile_w + ((int64_t)piece * NT + c0) * BM;
                unsigned long long *own = tile_x + ((int64_t)piece * NT + c0) * BM;
                const int ncols = B - c0 < 16 ? B - c0 : 16;
                if (piece != S - 1) {  // publish this piece
                    if (has_row && dbg_range(own_w, 15 * BM + 1, bd.xch, status))
                        xch::publish16(own, BM, v, ncols);
                    continue;
                }
                if (!has_row)
                    continue;  // (lanes 16-31 of an M = 64 tile; the warp reconverges above)
                // Reduce: pieces 0..S-2 in order, then this block's own piece.
                float sum[16];
                if (!dbg_range(tile_w + (int64_t)c0 * BM, (int64_t)(S - 1) * NT * BM + 15 * BM + 1, bd.xch, status)) {
                    ok = false;
                } else if (!(S > 3 ? xch::reduce16<4>(tile_x + (int64_t)c0 * BM, (int64_t)NT * BM, BM, S - 1, ncols, v,
                                                      own, sum, limit_ns)
                                   : xch::reduce16<2>(tile_x + (int64_t)c0 * BM, (int64_t)NT * BM, BM, S - 1, ncols, v,
                                                      own, sum, limit_ns))) {
                    record_status(status, DEP_DEV_TIMEOUT_EPILOGUE);
                    ok = false;
                }
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (j < ncols && mine && ok && dbg_ok((int64_t)(c0 + j) * N + n, bd.y, status))
                        y[(int64_t)(c0 + j) * N + n] = to_bf16(sum[j]);
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(acce0 + 8 * buf);
            buf ^= 1;
        }
    }

    __syncwarp();
    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after();
        tc::dealloc(tmem, Sh::TMEM_COLS);
    }
}

template <int NT, int BM>
size_t smem_bytes(int stages, int atoms)
{
    return split_smem_bytes(stages, atoms * SplitShape<NT, BM>::ATOM, SplitShape<NT, BM>::XFER_BYTES);
}

template <int NT, int BM>
cudaError_t prepare()
{
    static std::atomic<uint64_t> devices{0};
    return set_smem_attr(tc_split_kernel<NT, BM>, devices);
}

// Pieces actually used: never more than the k-tiles of a tile (no empty piece).
int64_t effective_splits(const dep_tactic_t &t, int64_t K)
{
    const int64_t KT = (K + t.tile_k - 1) / t.tile_k;
    return t.splits < KT ? t.splits : KT;
}

int64_t tiles_of(const dep_tactic_t &t, int64_t N)
{
    return (N + t.tile_n - 1) / t.tile_n;
}

template <int NT, int BM>
cudaError_t run_shape(const dep_tactic_t &t, const RunArgs &a)
{
    cudaError_t e = prepare<NT, BM>();
    if (e != cudaSuccess)
        return e;
    const int atoms = t.tile_k / kBK;
    // One copy per stage (a column-block view) when K is a multiple of 64; else
    // one per 64-column slice, whose tensor map zero-fills past column K.
    const int tma3 = a.K % kBK == 0;
    CUtensorMap tmW, tmX;
    if ((tma3 ? encode_bf16_3d_blocks(&tmW, a.W, (uint64_t)a.K, (uint64_t)a.N, BM, (uint32_t)atoms)
              : encode_bf16_2d(&tmW, a.W, (uint64_t)a.K, (uint64_t)a.N, kBK, BM, CU_TENSOR_MAP_SWIZZLE_128B)) !=
        CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int S = (int)effective_splits(t, a.K);
    const int64_t items = tiles_of(t, a.N) * S;
    const int grid = (int)(items < t.ctas ? items : t.ctas);
    const size_t smem = smem_bytes<NT, BM>(t.stages, atoms);
    int *dispenser = a.counters + a.n_counters - 2;
    for (int32_t r0 = 0; r0 < a.B; r0 += NT) {
        const int32_t rows = a.B - r0 < NT ? a.B - r0 : NT;
        const uint16_t *xr = a.x + (size_t)r0 * a.K;
        if ((tma3 ? encode_bf16_3d_blocks(&tmX, xr, (uint64_t)a.K, (uint64_t)rows, NT, (uint32_t)atoms)
                  : encode_bf16_2d(&tmX, xr, (uint64_t)a.K, (uint64_t)rows, kBK, NT, CU_TENSOR_MAP_SWIZZLE_128B)) !=
            CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        e = launch(tc_split_kernel<NT, BM>, dim3(grid), dim3(kThreads), smem, a.stream, a.pdl, tmW, tmX,
                   a.y + (size_t)r0 * a.N, rows, (int)a.N, (int)a.K, t.stages, atoms, S, tma3, a.xch, dispenser,
                   a.status, a.bounds(rows, smem), a.wait_limit_ns);
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

template <int NT, int BM>
int blocks_per_sm_shape(const dep_tactic_t &t)
{
    if (prepare<NT, BM>() != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, tc_split_kernel<NT, BM>, kThreads,
                                                      smem_bytes<NT, BM>(t.stages, t.tile_k / kBK)) != cudaSuccess)
        return 0;
    return n;
}

template <int NT, int BM>
size_t smem_shape(const dep_tactic_t &t)
{
    return smem_bytes<NT, BM>(t.stages, t.tile_k / kBK);
}

template <int NT, int BM>
cudaError_t prepare_shape(const dep_tactic_t &)
{
    return prepare<NT, BM>();
}

// The tactic's instantiation: MMA width (cols) x tile rows (tile_n).
#define DEP_TCS_DISPATCH(NAME, RET, FN, BAD)                                    \
    RET NAME(const dep_tactic_t &t)                                             \
    {                                                                           \
        const bool m64 = t.tile_n == 64;                                        \
        switch (t.cols) {                                                       \
        case 16: return m64 ? FN<16, 64>(t) : FN<16, 128>(t);                   \
        case 32: return m64 ? FN<32, 64>(t) : FN<32, 128>(t);                   \
        case 64: return m64 ? FN<64, 64>(t) : FN<64, 128>(t);                   \
        case 128: return m64 ? FN<128, 64>(t) : FN<128, 128>(t);                \
        case 256: return m64 ? FN<256, 64>(t) : FN<256, 128>(t);                \
        default: return BAD;                                                    \
        }                                                                       \
    }

DEP_TCS_DISPATCH(smem_for, size_t, smem_shape, 0)
DEP_TCS_DISPATCH(blocks_for, int, blocks_per_sm_shape, 0)
DEP_TCS_DISPATCH(prepare_for, cudaError_t, prepare_shape, cudaErrorInvalidValue)
#undef DEP_TCS_DISPATCH

// Self-test of the exchange's give-up path, on a plan's own regions: one warp
// publishes the words of pieces 1 and 3 of a 32-row, 16-column tile (as
// publishers would), then reduces pieces 0 and 1 with the exchange's reducer;
// piece 0 is never published, so the bounded wait gives up and the warp records
// DEP_DEV_TIMEOUT_EPILOGUE.  Piece 3's "full" flags stay behind, and so does a
// nonzero word at the start of the counters (where the split-K FMA kernel
// counts arrivals and the wide-batch kernel keeps its flags): the state a real
// give-up can leave a plan in.
__global__ void selftest_exchange_kernel(unsigned long long *xch, int *counters, int *status, uint64_t limit_ns)
{
    const int lane = threadIdx.x & 31;
    constexpr int64_t kCol = 32, kPiece = 16 * kCol;  // words [piece][column][row]
    uint32_t v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
        v[j] = __float_as_uint((float)(lane + j));
    xch::publish16(xch + kPiece + lane, kCol, v, 16);      // piece 1 published
    xch::publish16(xch + 3 * kPiece + lane, kCol, v, 16);  // piece 3: nobody reduces it
    __syncwarp();
    float out[16];
    if (!xch::reduce16(xch + lane, kPiece, kCol, 2, 16, v, xch + 2 * kPiece + lane, out, limit_ns))
        record_status(status, DEP_DEV_TIMEOUT_EPILOGUE);
    if (lane == 0)
        atomicExch(counters, 1);
}

}  // namespace

cudaError_t tcs_selftest_exchange(unsigned long long *xch, size_t xch_words, int *counters, int *status,
                                  uint64_t limit_ns, cudaStream_t stream)
{
    if (xch_words < 4 * 16 * 32)
        return cudaErrorInvalidValue;
    selftest_exchange_kernel<<<1, 32, 0, stream>>>(xch, counters, status, limit_ns);
    return cudaGetLastError();
}

bool tcs_valid(const dep_tactic_t &t)
{
    if (t.kind != DEP_KIND_TC_SPLIT || t.ctas < 1 || (t.tile_n != 64 && t.tile_n != 128))
        return false;  // MMA M = 64 or 128 weight rows
    if (t.tile_k != kBK && t.tile_k != 2 * kBK && t.tile_k != 4 * kBK)
        return false;  // 1, 2 or 4 slices of 64 columns per stage
    if (t.stages < 2 || t.stages > 16 || t.splits < 1 || t.splits > kMaxSplits)
        return false;
    const size_t smem = smem_for(t);
    return smem != 0 && smem <= (size_t)kMaxDynamicSmem;
}

size_t tcs_xch_words(const dep_tactic_t &t, int64_t N, int64_t K)
{
    const int64_t S = effective_splits(t, K);
    return S > 1 ? (size_t)tiles_of(t, N) * (size_t)S * (size_t)t.cols * (size_t)t.tile_n : 0;
}

size_t tcs_counters(const dep_tactic_t &, int64_t)
{
    return 2;  // the item counter pair at the end
}

int64_t tcs_items(const dep_tactic_t &t, int64_t N, int64_t K)
{
    return tiles_of(t, N) * effective_splits(t, K);
}

int tcs_blocks_per_sm(const dep_tactic_t &t)
{
    return blocks_for(t);
}

cudaError_t tcs_prepare_device()
{
    for (int32_t cols : {16, 32, 64, 128, 256})
        for (int32_t bm : {64, 128}) {
            dep_tactic_t t{};
            t.cols = cols;
            t.tile_n = bm;
            const cudaError_t e = prepare_for(t);
            if (e != cudaSuccess)
                return e;
        }
    return cudaSuccess;
}

cudaError_t tcs_run(const dep_tactic_t &t, const RunArgs &a)
{
    const bool m64 = t.tile_n == 64;
    switch (t.cols) {
    case 16: return m64 ? run_shape<16, 64>(t, a) : run_shape<16, 128>(t, a);
    case 32: return m64 ? run_shape<32, 64>(t, a) : run_shape<32, 128>(t, a);
    case 64: return m64 ? run_shape<64, 64>(t, a) : run_shape<64, 128>(t, a);
    case 128: return m64 ? run_shape<128, 64>(t, a) : run_shape<128, 128>(t, a);
    case 256: return m64 ? run_shape<256, 64>(t, a) : run_shape<256, 128>(t, a);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace dep
