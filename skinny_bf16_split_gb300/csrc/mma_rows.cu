// mma_rows.cu -- warp-level MMA tactic for small weights at up to 16 batch rows.
//
// Computes y[B,N] = BF16(x[B,K] . W[N,K]^T), BF16 products accumulated in FP32,
// at the batches of the split-K rows (runtime.hybrid page,
// HybridAttention.__init__: warp split-K up to 16 rows; runtime.dep page,
// DepProjection.run), for the shard-sized weights of a tensor-parallel
// deployment (runtime.hybrid page, projection_policies(tp, ...)).
//
// Why: on a 13-52 MB weight a call's fixed chain -- the preceding grid
// completes, the wait returns, x lands, the prefetched ring drains, pieces are
// exchanged, the blocks exit -- costs as much as streaming the weight.  The
// tcgen05 kinds hold tensor memory, which keeps them to one block per SM, so
// the next call's blocks cannot start streaming on an SM until the current
// call's block there has left.  This kernel holds no tensor memory: it
// multiplies with warp-level mma.sync (m16n8k16, BF16 in, FP32 accumulators in
// registers), takes a small ring, and so several blocks -- of this call and of
// the next, under programmatic dependent launch -- share an SM.
//
// Design (sm_103a):
//  * One block per tile of 16 weight rows sums the tile's whole K, or (splits
//    = 2 or 4, for long rows on few tiles) the S blocks of a thread-block
//    cluster each sum a contiguous piece of the 64-column slices and store
//    their 16 x 16 FP32 partials into rank 0's shared memory, which adds them
//    in rank order after a cluster barrier (no workspace either way).  Warp 0 lane 0 issues TMA copies: per stage a
//    box of `atoms` 64-column slices of the tile's 16 rows (one copy through the
//    column-block view when K % 64 == 0) and the same slices of x (16 rows,
//    rows past B zero), 128-byte swizzle.  Weight first, before waiting for the
//    preceding grid; x after.
//  * Warps 1-4 compute: warp w takes slice w of every stage (atoms = 4; with
//    atoms = 2, warps 1-2 take slices of even stages and 3-4 of odd ones), four
//    K steps of 16 per slice, two m16n8k16 MMAs per step (batch rows 0-7 and
//    8-15), A and B fragments read with ldmatrix from the swizzled slices.
//  * Each warp adds its slices in increasing K order; the four warps' 16 x 16
//    partials are added in warp order through shared memory, rounded to BF16
//    and stored.  Results depend on neither the grid nor timing.
//  * Every wait on a barrier is bounded in time.
#include <cuda_bf16.h>

#include "cluster.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace dep {
namespace {

constexpr int kBK = 64;              // columns per slice: one 128-byte swizzle row
constexpr int kTR = 16;              // weight rows per tile (MMA M)
constexpr int kXR = 16;              // batch rows per pass (two MMA N of 8)
constexpr int kComp = 4;             // compute warps
constexpr int kThreads = 32 * (1 + kComp);
constexpr int kSlice = kTR * kBK * 2;  // one weight slice: 2 KB (x slices are the same size)
constexpr int kMaxStages = 16;
constexpr int kMaxPieces = 4;        // K pieces of a tile: blocks of one cluster

__host__ __device__ constexpr int mr_stage(int atoms) { return 2 * atoms * kSlice; }
// Shared memory: the 1 KB-aligned ring (per stage: the weight slices, then the
// x slices), the four warps' partials, the K pieces' partials (rank 0 of a
// cluster), full[stages], empty[stages], the abort flag.
__host__ __device__ constexpr size_t mr_smem_bytes(int stages, int atoms)
{
    return 1024 + (size_t)stages * mr_stage(atoms) + (size_t)(kComp + kMaxPieces) * kTR * kXR * 4 +
           (size_t)2 * stages * 8 + 16;
}

// Four 8x8 BF16 matrices from shared memory (rows addressed per lane).
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// D (+)= A . B, m16n8k16, A row-major and B column-major BF16, FP32 accumulators.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Address of row r, 16-byte chunk c of a 16-row slice at `slice` (128-byte
// swizzle: chunk c of row r lies at chunk c ^ (r % 8)).
__device__ __forceinline__ uint32_t swz(uint32_t slice, int r, int c)
{
    return slice + (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// Store into the shared memory of a CTA of this cluster (a mapped address).
__device__ __forceinline__ void st_cluster_f32(uint32_t a, float v)
{
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

// Compute warps only (named barrier 1).
__device__ __forceinline__ void comp_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kComp) : "memory");
}

__global__ void __launch_bounds__(kThreads)
    mma_rows_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                    uint16_t *__restrict__ y, int B, int N, int K, int stages, int atoms, int tma3, int S,
                    int *__restrict__ status, const Bounds bd, uint64_t limit_ns)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle boxes need 1 KB alignment
    uint8_t *smem = smem_raw + (base - raw);
    if (!dbg_ok((base - raw) + mr_smem_bytes(stages, atoms) - 1024 - 1, bd.smem, status))
        return;
    const int STAGE = mr_stage(atoms), XOFF = atoms * kSlice;
    float *part = reinterpret_cast<float *>(smem + (size_t)stages * STAGE);  // [warp][row][batch row]
    float *red = part + kComp * kTR * kXR;                                    // [piece][row][batch row]
    uint64_t *bars = reinterpret_cast<uint64_t *>(red + kMaxPieces * kTR * kXR);
    const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * stages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 2 * stages);

    // With S > 1 the S blocks of a cluster share a tile: rank r sums the
    // 64-column slices [r KT / S, (r + 1) KT / S) and rank 0 adds the pieces.
    const int rank = S > 1 ? (int)cluster_rank() : 0;
    const int KT_ALL = (K + kBK - 1) / kBK;
    const int S0 = rank * KT_ALL / S;                   // this block's first slice
    const int KT = (rank + 1) * KT_ALL / S - S0;        // its slices
    const int KS = (KT + atoms - 1) / atoms;            // stages
    const int row0 = (int)(blockIdx.x / (unsigned)S) * kTR;  // the tile
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto slices_of = [&](int k) { return KT - k * atoms < atoms ? KT - k * atoms : atoms; };
    const int pre = KS < stages ? KS : stages;

    uint64_t pol_w = 0, pol_x = 0;
    auto issue_w = [&](int st, int k) {
        const uint32_t dst = base + (uint32_t)(st * STAGE), bar = full0 + 8 * st;
        const int na = slices_of(k);
        mbar_arrive_expect_tx(bar, (uint32_t)((tma3 ? atoms : na) * 2 * kSlice));  // weight and x
        if (tma3) {
            tma_load_3d(dst, &tmW, 0, row0, S0 + k * atoms, bar, pol_w);
        } else {
            for (int a = 0; a < na; ++a)
                tma_load_2d(dst + (uint32_t)(a * kSlice), &tmW, (S0 + k * atoms + a) * kBK, row0, bar, pol_w);
        }
    };
    auto issue_x = [&](int st, int k) {
        const uint32_t dst = base + (uint32_t)(st * STAGE + XOFF), bar = full0 + 8 * st;
        if (tma3) {
            tma_load_3d(dst, &tmX, 0, 0, S0 + k * atoms, bar, pol_x);
        } else {
            for (int a = 0; a < slices_of(k); ++a)
                tma_load_2d(dst + (uint32_t)(a * kSlice), &tmX, (S0 + k * atoms + a) * kBK, 0, bar, pol_x);
        }
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < stages; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, kComp);
        }
        *abort_flag = 0;
        fence_mbar_init();
        griddep_launch_dependents();
        // The weight is not written by preceding work: fill the ring first.
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmX);
        pol_w = policy_evict_first();
        pol_x = policy_evict_last();
        for (int i = 0; i < pre; ++i)
            issue_w(i, i);
    }
    __syncthreads();
    if (S > 1)
        cluster_sync();  // every block of the cluster has started

    // Epilogue state of a compute thread: its batch row, first weight row, sums.
    int en = 0, er = 0;
    float ev[2] = {0.f, 0.f};
    bool eok = false;
    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            griddep_wait();  // x may be written by the preceding grid
            for (int i = 0; i < pre; ++i)
                issue_x(i, i);
            int s = pre % stages;
            uint32_t ph = pre == stages ? 1u : 0u;
            int64_t issued = pre;
            for (int k = pre; k < KS; ++k) {
                if (*abort_flag)
                    break;
                if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, limit_ns)) {
                    record_status(status, DEP_DEV_TIMEOUT_PRODUCER);
                    *abort_flag = 1;
                    break;
                }
                issue_w(s, k);
                issue_x(s, k);
                ++issued;
                if (++s == stages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
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
    } else {
        // ---------------- compute warps ----------------
        const int w = warp - 1;
        float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};  // batch rows 0-7, 8-15
        // ldmatrix row addresses of this lane: A (weight) row and chunk half,
        // B (x) batch row and chunk half.
        const int ar = lane & 15, ah = lane >> 4;
        const int bn = (lane & 7) + ((lane >> 4) << 3), bh = (lane >> 3) & 1;
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int k = 0; k < KS; ++k) {
            const bool got = !*abort_flag && mbar_wait(full0 + 8 * s, ph, limit_ns);
            if (!__all_sync(0xffffffffu, got)) {
                if (!*abort_flag)
                    record_status(status, DEP_DEV_TIMEOUT_MMA);
                *abort_flag = 1;
                ok = false;
                break;
            }
            const uint32_t sa = base + (uint32_t)(s * STAGE);
            const int na = slices_of(k);
            for (int a = 0; a < na; ++a) {
                if (((k * atoms + a) & (kComp - 1)) != w)
                    continue;  // slice g of the call goes to warp g % 4
                const uint32_t ws = sa + (uint32_t)(a * kSlice), xs = sa + (uint32_t)(XOFF + a * kSlice);
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
                    ldmatrix_x4(swz(ws, ar, 2 * kk + ah), a0, a1, a2, a3);
                    ldmatrix_x4(swz(xs, bn, 2 * kk + bh), b0, b1, b2, b3);
                    mma_16816(acc0, a0, a1, a2, a3, b0, b1);
                    mma_16816(acc1, a0, a1, a2, a3, b2, b3);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(empty0 + 8 * s);  // this warp is done with the stage
            if (++s == stages) {
                s = 0;
                ph ^= 1u;
            }
        }
        // The four warps' partials in shared memory, then added in warp order.
        {
            float *p = part + w * kTR * kXR;
            const int r = lane >> 2, c = 2 * (lane & 3);
            p[r * kXR + c] = acc0[0];
            p[r * kXR + c + 1] = acc0[1];
            p[(r + 8) * kXR + c] = acc0[2];
            p[(r + 8) * kXR + c + 1] = acc0[3];
            p[r * kXR + 8 + c] = acc1[0];
            p[r * kXR + 8 + c + 1] = acc1[1];
            p[(r + 8) * kXR + 8 + c] = acc1[2];
            p[(r + 8) * kXR + 8 + c + 1] = acc1[3];
        }
        comp_sync();
        const int t = threadIdx.x - 32;          // 0..127
        en = t >> 3;                             // batch row
        er = 2 * (t & 7);                        // first of two weight rows
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int i = (er + j) * kXR + en;
            ev[j] = ((part[i] + part[kTR * kXR + i]) + part[2 * kTR * kXR + i]) + part[3 * kTR * kXR + i];
        }
        eok = ok;
        if (S > 1) {  // this block's piece into rank 0's slot `rank`
#pragma unroll
            for (int j = 0; j < 2; ++j)
                st_cluster_f32(peer_addr(smem_u32(red + (rank * kTR + er + j) * kXR + en), 0u), ev[j]);
        }
    }
    if (S > 1) {
        cluster_sync();  // the pieces are in rank 0; no block leaves while another may write into it
        if (rank == 0 && warp >= 1) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {  // the pieces in rank order
                float v = red[(er + j) * kXR + en];
                for (int p = 1; p < S; ++p)
                    v = v + red[(p * kTR + er + j) * kXR + en];
                ev[j] = v;
            }
        }
    }
    if (warp >= 1 && rank == 0 && eok && en < B && row0 + er < N) {
        griddep_wait();  // y may still be in use by the preceding grid
        uint16_t *yr = y + (int64_t)en * N + row0 + er;
        const bool two = row0 + er + 1 < N;
        if (two && (N & 1) == 0 && dbg_ok((int64_t)en * N + row0 + er + 1, bd.y, status)) {
            *reinterpret_cast<uint32_t *>(yr) = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(ev[0])) |
                                                ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(ev[1])) << 16);
        } else {
            if (dbg_ok((int64_t)en * N + row0 + er, bd.y, status))
                yr[0] = __bfloat16_as_ushort(__float2bfloat16_rn(ev[0]));
            if (two && dbg_ok((int64_t)en * N + row0 + er + 1, bd.y, status))
                yr[1] = __bfloat16_as_ushort(__float2bfloat16_rn(ev[1]));
        }
    }
}

}  // namespace
}  // namespace dep

namespace dep {
namespace {

cudaError_t prepare()
{
    static std::atomic<uint64_t> devices{0};
    return set_smem_attr(mma_rows_kernel, devices);
}

}  // namespace

bool mma_rows_valid(const dep_tactic_t &t)
{
    if (t.kind != DEP_KIND_WARP_MMA || t.ctas < 1 || t.tile_n != kTR || t.cols != kXR)
        return false;  // tiles of 16 weight rows, passes of 16 batch rows
    if (t.splits != 0 && t.splits != 1 && t.splits != 2 && t.splits != kMaxPieces)
        return false;  // K pieces per tile: 1 (0), 2 or 4 blocks of a cluster
    if (t.tile_k != kBK && t.tile_k != 2 * kBK && t.tile_k != 4 * kBK)
        return false;  // 1, 2 or 4 slices of 64 columns per stage
    if (t.stages < 2 || t.stages > kMaxStages)
        return false;
    return mr_smem_bytes(t.stages, t.tile_k / kBK) <= (size_t)kMaxDynamicSmem;
}

int64_t mma_rows_tiles(const dep_tactic_t &t, int64_t N)
{
    return (N + kTR - 1) / kTR * (t.splits > 1 ? t.splits : 1);  // blocks of a launch
}

cudaError_t mma_rows_prepare_device()
{
    return prepare();
}

cudaError_t mma_rows_run(const dep_tactic_t &t, const RunArgs &a)
{
    cudaError_t e = prepare();
    if (e != cudaSuccess)
        return e;
    const int atoms = t.tile_k / kBK;
    // One copy per stage (column-block views) when K is a multiple of 64; else
    // one per 64-column slice, whose 2-D maps zero-fill past column K.
    const int tma3 = a.K % kBK == 0;
    CUtensorMap tmW, tmX;
    if ((tma3 ? encode_bf16_3d_blocks(&tmW, a.W, (uint64_t)a.K, (uint64_t)a.N, kTR, (uint32_t)atoms)
              : encode_bf16_2d(&tmW, a.W, (uint64_t)a.K, (uint64_t)a.N, kBK, kTR, CU_TENSOR_MAP_SWIZZLE_128B)) !=
        CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int64_t T = (a.N + kTR - 1) / kTR;  // tiles
    const size_t smem = mr_smem_bytes(t.stages, atoms);
    // K pieces per tile, each at least one 64-column slice
    const int64_t KT = (a.K + kBK - 1) / kBK;
    int S = t.splits > 1 ? t.splits : 1;
    while (S > 1 && KT < S)
        S /= 2;
    for (int32_t r0 = 0; r0 < a.B; r0 += kXR) {
        const int32_t rows = a.B - r0 < kXR ? a.B - r0 : kXR;
        const uint16_t *xr = a.x + (size_t)r0 * a.K;
        if ((tma3 ? encode_bf16_3d_blocks(&tmX, xr, (uint64_t)a.K, (uint64_t)rows, kXR, (uint32_t)atoms)
                  : encode_bf16_2d(&tmX, xr, (uint64_t)a.K, (uint64_t)rows, kBK, kXR, CU_TENSOR_MAP_SWIZZLE_128B)) !=
            CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(T * S));  // one block per tile and K piece
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = a.stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = a.pdl ? 1 : 0;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)S;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = S > 1 ? 2 : 1;
        e = cudaLaunchKernelEx(&cfg, mma_rows_kernel, tmW, tmX, a.y + (size_t)r0 * a.N, (int)rows, (int)a.N,
                               (int)a.K, t.stages, atoms, tma3, S, a.status, a.bounds(rows, smem), a.wait_limit_ns);
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

}  // namespace dep
