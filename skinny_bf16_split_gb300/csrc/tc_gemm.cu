// tc_gemm.cu -- tcgen05 tensor-core tactic for the decode projection.
//
// Computes y[B,N] = BF16(x[B,K] . W[N,K]^T), BF16 products accumulated in FP32,
// for the batches where the FMA pipe would be the bottleneck (runtime.hybrid
// page, HybridAttention.__init__: past the split-K rows the projection runs the
// stock FP32-accumulated BF16 GEMM; runtime.dep page, DepProjection).
//
// Design (sm_103a, one CTA per SM, no clusters, no multicast):
//  * Swap-AB: the MMA's M side is 128 weight rows, its N side the batch padded
//    to NT (16..256), so one weight tile feeds one MMA and a tiny batch wastes
//    only tensor throughput, never weight bytes.  D[128 x NT] lives in TMEM.
//  * Work units are (128-row tile, tile_k-column k-tile) pairs, tile_k = 64, 128
//    or 256; the persistent blocks take equal contiguous ranges (stream-K),
//    exactly as the FMA tactic.
//  * Warp 0: TMA producer.  Per stage, tile_k / 64 weight slices [128 x 64] and
//    activation slices [NT x 64] land in a shared-memory ring in the 128-byte
//    swizzle layout (wider stages give each weight row longer contiguous reads).
//  * Warp 1: allocates TMEM (two accumulator buffers), one thread issues
//    tcgen05.mma (4 per 64-column slice, K = 16 each) and releases each stage with
//    tcgen05.commit; at the end of a segment it commits the accumulator.  One
//    thread issues an MMA only about every 67 cycles, whatever its M and N (up
//    to N = 128): too little work per instruction at N <= 32 to drain a full
//    ring quickly.  There warp 2 issues too: issuer i takes a fixed half of
//    every stage's K steps into its own accumulator, and the epilogue adds the
//    two in issuer order (FP32, deterministic; the K-piece kernel uses the same
//    rule, so the two kernels' sums of one tile agree bit for bit).
//  * Warps 3-6: epilogue.  Each owns the 32 TMEM lanes (= weight rows) of its
//    quadrant, reads its accumulator with tcgen05.ld, frees it for the MMA of
//    the next-but-one segment, and either stores BF16 y (segment = whole tile)
//    or exchanges FP32 partials for the split-K reduction through flagged
//    64-bit words (exchange.cuh).  Every block publishes at most one piece (in
//    its slot 0): the segment of a split tile whose last unit it does not own.
//    The block owning the tile's last unit reduces, adding the pieces in
//    increasing block order with its own last (kept in its slot 1 for
//    inspection).  The other blocks meet that tile as the last tile of their
//    range, which they visit first, so they publish before doing anything else
//    and never wait: no deadlock, and the reducer's words are usually ready
//    when it gets there.  No float atomics: results are identical from run to
//    run.
//  * Every wait is bounded in time; on a give-up the block records a code,
//    lets every role finish, waits for its MMAs and copies, and frees TMEM.
#include <cuda_bf16.h>

#include "exchange.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace dep {
namespace {

constexpr int kBM = 128;          // weight rows per tile (MMA M)
constexpr int kBK = 64;           // columns per stage: one 128-byte swizzle row
constexpr int kUmmaK = 16;        // K of one kind::f16 MMA
constexpr int kThreads = 224;     // warp 0 TMA, warps 1-2 MMA (warp 1 owns TMEM), warps 3-6 epilogue
constexpr int kEpiWarps = 4;
constexpr int kABytes = kBM * kBK * 2;  // 16 KB weight tile per stage

// A stage holds `atoms` consecutive 64-column slices of one unit: the weight
// slices [128 x 64] first (16 KB each), then the activation slices [NT x 64].
template <int NT>
struct TcShape {
    static constexpr int B_BYTES = NT * kBK * 2;     // one activation slice (a multiple of 1024)
    static constexpr int ATOM = kABytes + B_BYTES;   // bytes per 64-column slice pair
    static constexpr int ISSUERS = NT <= 32 ? 2 : 1;  // MMA issuers, one accumulator each per buffer
    static constexpr uint32_t TMEM_COLS = 2 * ISSUERS * NT < 32 ? 32 : 2 * ISSUERS * NT;
};

__device__ __forceinline__ uint16_t to_bf16(float v)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   uint16_t *__restrict__ y, int B, int N, int K, int stages, int atoms, int tma3,
                   unsigned long long *__restrict__ xch, int *__restrict__ status, const Bounds bd,
                   uint64_t limit_ns)
{
    using S = TcShape<NT>;
    const int STAGE = atoms * S::ATOM;   // bytes per stage
    const int KG = atoms * kBK;          // columns per unit
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle tiles need 1 KB alignment
    uint8_t *smem = smem_raw + (base - raw);
    if (!dbg_ok((base - raw) + (size_t)stages * STAGE + (2 * (size_t)stages + 5) * 8 + 8 - 1, bd.smem, status))
        return;  // the ring, the barriers and the TMEM slot must lie in the launch's shared memory
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)stages * STAGE);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = full0 + 8 * stages;
    const uint32_t accf0 = empty0 + 8 * stages;  // accumulator ready, 2 buffers
    const uint32_t acce0 = accf0 + 16;           // accumulator drained, 2 buffers
    const uint32_t done = acce0 + 16;            // all MMAs complete
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * stages + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int64_t T = (N + kBM - 1) / kBM, KTILES = (K + KG - 1) / KG, U = T * KTILES;
    const int64_t C = gridDim.x, c = blockIdx.x;
    const int64_t u_begin = sk_begin(c, U, C), u_end = sk_begin(c + 1, U, C);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, S::ISSUERS);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, S::ISSUERS);
            mbar_init(acce0 + 8 * b, kEpiWarps);
        }
        mbar_init(done, S::ISSUERS);
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
            // The weight is not written by preceding work: fill the ring with its
            // first tiles, then wait for the preceding grid before reading x.
            const SegOrder order(u_begin, u_end, KTILES);
            const int64_t pre = (u_end - u_begin) < stages ? (u_end - u_begin) : stages;
            UnitCursor cur(order);
            for (int64_t i = 0; i < pre; ++i, cur.next()) {
                const int64_t u = cur.u;
                const uint32_t st = base + (uint32_t)(i * STAGE);
                mbar_arrive_expect_tx(full0 + 8 * (int)i, STAGE);
                if (tma3)  // the stage's slices in one copy (column-block view of W)
                    tma_load_3d(st, &tmW, 0, (int)(u / KTILES) * kBM, (int)(u % KTILES) * atoms, full0 + 8 * (int)i,
                                pol_w);
                else
                    for (int a = 0; a < atoms; ++a)
                        tma_load_2d(st + (uint32_t)(a * kABytes), &tmW, (int)(u % KTILES) * KG + a * kBK,
                                    (int)(u / KTILES) * kBM, full0 + 8 * (int)i, pol_w);
            }
            griddep_wait();
            UnitCursor cx(order);
            for (int64_t i = 0; i < pre; ++i, cx.next()) {
                const int64_t u = cx.u;
                const uint32_t xs = base + (uint32_t)(i * STAGE) + (uint32_t)(atoms * kABytes);
                if (tma3)
                    tma_load_3d(xs, &tmX, 0, 0, (int)(u % KTILES) * atoms, full0 + 8 * (int)i, pol_x);
                else
                    for (int a = 0; a < atoms; ++a)
                        tma_load_2d(xs + (uint32_t)(a * S::B_BYTES), &tmX, (int)(u % KTILES) * KG + a * kBK, 0,
                                    full0 + 8 * (int)i, pol_x);
            }
            int s = (int)(pre % stages);
            uint32_t ph = pre == stages ? 1u : 0u;
            int64_t issued = pre;
            for (; !cur.done(); cur.next()) {
                const int64_t u = cur.u;
                if (*abort_flag)
                    break;
                if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, limit_ns)) {
                    record_status(status, DEP_DEV_TIMEOUT_PRODUCER);
                    *abort_flag = 1;
                    break;
                }
                const uint32_t st = base + (uint32_t)(s * STAGE);
                mbar_arrive_expect_tx(full0 + 8 * s, STAGE);
                const int t = (int)(u / KTILES), kg = (int)(u % KTILES);
                if (tma3) {
                    tma_load_3d(st, &tmW, 0, t * kBM, kg * atoms, full0 + 8 * s, pol_w);
                    tma_load_3d(st + (uint32_t)(atoms * kABytes), &tmX, 0, 0, kg * atoms, full0 + 8 * s, pol_x);
                } else {
                    for (int a = 0; a < atoms; ++a)
                        tma_load_2d(st + (uint32_t)(a * kABytes), &tmW, kg * KG + a * kBK, t * kBM, full0 + 8 * s,
                                    pol_w);
                    for (int a = 0; a < atoms; ++a)
                        tma_load_2d(st + (uint32_t)(atoms * kABytes + a * S::B_BYTES), &tmX, kg * KG + a * kBK, 0,
                                    full0 + 8 * s, pol_x);
                }
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
    } else if (warp == 1 || warp == 2) {
        // ---------------- MMA issuers ----------------
        // Issuer mi takes K steps [mi H, (mi + 1) H) of every stage (H = the
        // stage's steps / issuers) into its own accumulator of each buffer.
        const int mi = warp - 1;
        if (lane == 0 && mi < S::ISSUERS) {
            constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, NT);
            const int H = atoms * (kBK / kUmmaK) / S::ISSUERS;
            int s = 0;
            uint32_t ph = 0, acce_ph = 0;
            int buf = 0;
            const SegOrder order(u_begin, u_end, KTILES);
            bool ok = true;
            for (int64_t seg = 0; seg < order.m && ok; ++seg) {
                const int64_t t = order.tile(seg);
                const int64_t seg_end = order.seg_end(t);
                int64_t u = order.seg_begin(t);
                if (!mbar_wait(acce0 + 8 * buf, ((acce_ph >> buf) & 1u) ^ 1u, limit_ns)) {
                    record_status(status, DEP_DEV_TIMEOUT_MMA);
                    *abort_flag = 1;
                    break;
                }
                acce_ph ^= 1u << buf;
                tc::fence_after();
                const uint32_t d = tmem + (uint32_t)((buf * S::ISSUERS + mi) * NT);
                uint32_t accumulate = 0;
                for (; u < seg_end; ++u) {
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
                    tc::mma_stage<kABytes, S::B_BYTES>(d, st, st + (uint32_t)(atoms * kABytes), mi * H, H, idesc,
                                                       accumulate);
                    tc::commit(empty0 + 8 * s);  // the stage is free once every issuer's MMAs finish
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok)
                    break;
                tc::commit(accf0 + 8 * buf);  // the accumulator is final once every issuer's MMAs finish
                buf ^= 1;
            }
            tc::commit(done);  // TMEM is freed at the end: wait for every MMA
            if (!mbar_wait(done, 0, limit_ns))
                record_status(status, DEP_DEV_TIMEOUT_MMA);
        }
    } else {
        // ---------------- epilogue warps ----------------
        griddep_wait();  // the exchange words and y may still be in use by the preceding grid
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const int row = 32 * q + lane;
        uint32_t accf_ph = 0;
        int buf = 0;
        const SegOrder order(u_begin, u_end, KTILES);
        for (int64_t seg = 0; seg < order.m; ++seg) {
            const int64_t t = order.tile(seg);
            const bool whole = (order.seg_begin(t) == t * KTILES) && (order.seg_end(t) == (t + 1) * KTILES);
            if (!mbar_wait(accf0 + 8 * buf, (accf_ph >> buf) & 1u, limit_ns)) {
                record_status(status, DEP_DEV_TIMEOUT_EPILOGUE);
                *abort_flag = 1;
                break;
            }
            accf_ph ^= 1u << buf;
            tc::fence_after();
            const int64_t n = t * kBM + row;
            // buffer buf's accumulators: issuer 0's, then issuer 1's (NT columns each)
            const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * S::ISSUERS * NT);
            // Pieces of tile t: the segments of blocks c_first..c_last, in block order.
            // Exchange words: [block][slot][b][row]; slot 0 published, slot 1 own.
            const int64_t c_first = sk_owner(t * KTILES, U, C);
            const int64_t c_last = sk_owner(t * KTILES + KTILES - 1, U, C);
            bool ok = true;
#pragma unroll 1
            for (int c0 = 0; c0 < NT && c0 < B; c0 += 16) {
                __syncwarp();  // tcgen05.ld is warp-collective: every lane, converged
                uint32_t v[16], v1[16];
                tc::ld16(taddr + (uint32_t)c0, v);
                if (S::ISSUERS == 2)
                    tc::ld16(taddr + (uint32_t)(NT + c0), v1);
                tc::wait_ld();
                if (S::ISSUERS == 2) {  // the block's partial: issuer 0's half of K, then issuer 1's
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(v1[j]));
                }
                const int ncols = B - c0 < 16 ? B - c0 : 16;
                if (whole) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (j < ncols && n < N && dbg_ok((int64_t)(c0 + j) * N + n, bd.y, status))
                            y[(int64_t)(c0 + j) * N + n] = to_bf16(__uint_as_float(v[j]));
                    continue;
                }
                if (c != c_last) {  // publish this block's piece
                    const int64_t w0 = ((c * 2) * NT + c0) * kBM + row;
                    if (dbg_range(w0, 15 * kBM + 1, bd.xch, status))
                        xch::publish16(xch + w0, kBM, v, ncols);
                    continue;
                }
                float sum[16];
                const int64_t r0 = ((c_first * 2) * NT + c0) * kBM + row, own0 = ((c * 2 + 1) * NT + c0) * kBM + row;
                if (!dbg_range(r0, (c_last - c_first - 1) * 2 * (int64_t)NT * kBM + 15 * kBM + 1, bd.xch, status) ||
                    !dbg_range(own0, 15 * kBM + 1, bd.xch, status)) {
                    ok = false;
                } else if (!xch::reduce16(xch + r0, 2 * (int64_t)NT * kBM, kBM, (int)(c_last - c_first), ncols, v,
                                          xch + own0, sum, limit_ns)) {
                    record_status(status, DEP_DEV_TIMEOUT_EPILOGUE);
                    ok = false;
                }
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (j < ncols && n < N && ok && dbg_ok((int64_t)(c0 + j) * N + n, bd.y, status))
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
        tc::dealloc(tmem, S::TMEM_COLS);
    }
}

constexpr size_t kMaxSmem = kMaxDynamicSmem;

template <int NT>
size_t smem_bytes(int stages, int atoms)
{
    return 1024 + (size_t)stages * atoms * TcShape<NT>::ATOM + (size_t)(2 * stages + 5) * 8 + 16;
}

template <int NT>
cudaError_t prepare()
{
    static std::atomic<uint64_t> devices{0};
    return set_smem_attr(tc_gemm_kernel<NT>, devices);
}

template <int NT>
cudaError_t run_nt(const dep_tactic_t &t, const RunArgs &a)
{
    cudaError_t e = prepare<NT>();
    if (e != cudaSuccess)
        return e;
    const int atoms = t.tile_k / kBK;
    // One copy per stage (a column-block view) when K is a multiple of 64; else
    // one per 64-column slice, whose tensor map zero-fills past column K.
    const int tma3 = a.K % kBK == 0;
    CUtensorMap tmW, tmX;
    if ((tma3 ? encode_bf16_3d_blocks(&tmW, a.W, (uint64_t)a.K, (uint64_t)a.N, kBM, (uint32_t)atoms)
              : encode_bf16_2d(&tmW, a.W, (uint64_t)a.K, (uint64_t)a.N, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B)) !=
        CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int64_t T = (a.N + kBM - 1) / kBM, KT = (a.K + t.tile_k - 1) / t.tile_k, U = T * KT;
    const int grid = (int)(U < t.ctas ? U : t.ctas);
    const size_t smem = smem_bytes<NT>(t.stages, atoms);
    for (int32_t r0 = 0; r0 < a.B; r0 += NT) {
        const int32_t rows = a.B - r0 < NT ? a.B - r0 : NT;
        const uint16_t *xr = a.x + (size_t)r0 * a.K;
        if ((tma3 ? encode_bf16_3d_blocks(&tmX, xr, (uint64_t)a.K, (uint64_t)rows, NT, (uint32_t)atoms)
                  : encode_bf16_2d(&tmX, xr, (uint64_t)a.K, (uint64_t)rows, kBK, NT, CU_TENSOR_MAP_SWIZZLE_128B)) !=
            CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        e = launch(tc_gemm_kernel<NT>, dim3(grid), dim3(kThreads), smem, a.stream, a.pdl, tmW, tmX,
                   a.y + (size_t)r0 * a.N, rows, (int)a.N, (int)a.K, t.stages, atoms, tma3, a.xch, a.status,
                   a.bounds(rows, smem), a.wait_limit_ns);
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

template <int NT>
int blocks_per_sm(int stages, int atoms)
{
    if (prepare<NT>() != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, tc_gemm_kernel<NT>, kThreads,
                                                      smem_bytes<NT>(stages, atoms)) != cudaSuccess)
        return 0;
    return n;
}

size_t smem_for(const dep_tactic_t &t)
{
    const int atoms = t.tile_k / kBK;
    switch (t.cols) {
    case 16: return smem_bytes<16>(t.stages, atoms);
    case 32: return smem_bytes<32>(t.stages, atoms);
    case 64: return smem_bytes<64>(t.stages, atoms);
    case 128: return smem_bytes<128>(t.stages, atoms);
    case 256: return smem_bytes<256>(t.stages, atoms);
    default: return 0;
    }
}

}  // namespace

bool tc_valid(const dep_tactic_t &t)
{
    if (t.kind != DEP_KIND_TC || t.ctas < 1 || t.tile_n != kBM)
        return false;
    if (t.tile_k != kBK && t.tile_k != 2 * kBK && t.tile_k != 4 * kBK)
        return false;  // 1, 2 or 4 slices of 64 columns per stage
    if (t.stages < 2 || t.stages > 16)
        return false;
    const size_t smem = smem_for(t);
    return smem != 0 && smem <= kMaxSmem;
}

int64_t tc_units(const dep_tactic_t &t, int64_t N, int64_t K)
{
    return ((N + kBM - 1) / kBM) * ((K + t.tile_k - 1) / t.tile_k);
}

size_t tc_xch_words_per_cta(const dep_tactic_t &t)
{
    return 2 * (size_t)t.cols * kBM;  // slot 0 published piece, slot 1 own piece
}

size_t tc_xch_words(const dep_tactic_t &t, int64_t N, int64_t K)
{
    const int64_t T = (N + kBM - 1) / kBM, U = tc_units(t, N, K);
    const int64_t C = U < t.ctas ? U : t.ctas;
    return C == T ? 0 : (size_t)C * tc_xch_words_per_cta(t);  // one block per tile: no split
}

int tc_blocks_per_sm(const dep_tactic_t &t)
{
    const int atoms = t.tile_k / kBK;
    switch (t.cols) {
    case 16: return blocks_per_sm<16>(t.stages, atoms);
    case 32: return blocks_per_sm<32>(t.stages, atoms);
    case 64: return blocks_per_sm<64>(t.stages, atoms);
    case 128: return blocks_per_sm<128>(t.stages, atoms);
    case 256: return blocks_per_sm<256>(t.stages, atoms);
    default: return 0;
    }
}

cudaError_t tc_prepare_device()
{
    for (cudaError_t e : {prepare<16>(), prepare<32>(), prepare<64>(), prepare<128>(), prepare<256>()})
        if (e != cudaSuccess)
            return e;
    return cudaSuccess;
}

cudaError_t tc_run(const dep_tactic_t &t, const RunArgs &a)
{
    switch (t.cols) {
    case 16: return run_nt<16>(t, a);
    case 32: return run_nt<32>(t, a);
    case 64: return run_nt<64>(t, a);
    case 128: return run_nt<128>(t, a);
    case 256: return run_nt<256>(t, a);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace dep
