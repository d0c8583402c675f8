// api.cpp -- the C ABI: plans (tactic tables), validation and dispatch.
//
// A plan mirrors DepProjection.__init__ (runtime.dep page): it is built once per
// weight shape and batch set and keeps a table keyed by "max rows"; a batch takes
// the entry of the smallest key >= B, else of the largest key (runtime.dep page,
// _bins).  The run call mirrors DepProjection.run: it writes the projection into
// the caller's preallocated output.
#include <algorithm>
#include <cerrno>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "internal.h"

using dep::RunArgs;

struct dep_plan_s {
    int64_t N = 0, K = 0;
    bool host_only = true;
    int device = -1;
    int sm_count = 0;
    std::string device_name;
    std::vector<dep_tactic_t> table;  // sorted by max_rows, unique keys
    void *dev_block = nullptr;        // one allocation, carved below
    size_t dev_bytes = 0;
    int *status = nullptr;
    int *counters = nullptr;
    size_t n_counters = 0;
    float *ws = nullptr;
    size_t ws_floats = 0;
    unsigned long long *xch = nullptr;  // K-piece exchange words, zeroed at allocation
    size_t xch_words = 0;
    uint16_t *x_stage = nullptr;
    uint16_t *y_stage = nullptr;
    int32_t stage_rows = 0;
    uint64_t wait_limit_ns = 1000000000ull;  // 1 s per wait
    bool fault_launch = false;
    bool log = false;
    bool pdl = false;  // DEP_PLAN_PDL
    bool keep_pieces = false;  // DEP_PLAN_KEEP_PIECES
};

namespace {

const int32_t kDefaultBatches[] = {1, 2, 4, 8, 16, 32, 64, 128, 256};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void *a, size_t abytes, const void *b, size_t bbytes)
{
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

bool env_is(const char *name, const char *value)
{
    const char *v = std::getenv(name);
    return v && std::strcmp(v, value) == 0;
}

int32_t pow2_at_least(int32_t b)
{
    int32_t p = 1;
    while (p < b)
        p <<= 1;
    return p;
}

bool tactic_valid(const dep_tactic_t &t)
{
    if (t.max_rows < 1)
        return false;
    if (t.kind == DEP_KIND_TC_SPLIT)
        return dep::tcs_valid(t);
    if (t.kind == DEP_KIND_TC_WIDE)
        return dep::wide_valid(t);
    if (t.kind == DEP_KIND_TC_CLUSTER)
        return dep::cluster_valid(t);
    if (t.kind == DEP_KIND_TC_XM)
        return dep::xm_valid(t);
    if (t.kind == DEP_KIND_WARP_MMA)
        return dep::mma_rows_valid(t);
    if (t.splits != 0)
        return false;  // only the K-piece tactic has pieces
    if (t.kind == DEP_KIND_SPLITK_FMA)
        return dep::fma_valid(t);
    if (t.kind == DEP_KIND_TC)
        return dep::tc_valid(t);
    if (t.kind == DEP_KIND_ROWS)
        return dep::rows_valid(t);
    return false;
}

size_t ws_per_cta(const dep_tactic_t &t)
{
    switch (t.kind) {
    case DEP_KIND_SPLITK_FMA: return dep::fma_ws_per_cta(t);
    case DEP_KIND_TC_WIDE: return dep::wide_ws_per_cta(t);
    default: return 0;  // whole rows: no partials; other tensor-core kinds: exchange words instead
    }
}

// Blocks a launch really uses: never more than the work units (stream-K) or tiles.
int64_t effective_ctas(const dep_tactic_t &t, int64_t N, int64_t K)
{
    const int64_t U = t.kind == DEP_KIND_SPLITK_FMA ? dep::fma_units(t, N, K)
                      : t.kind == DEP_KIND_TC       ? dep::tc_units(t, N, K)
                      : t.kind == DEP_KIND_TC_WIDE  ? dep::wide_units(t, N, K)
                      : t.kind == DEP_KIND_TC_XM    ? dep::xm_tiles(t, N)
                      : t.kind == DEP_KIND_WARP_MMA ? dep::mma_rows_tiles(t, N)
                                                    : dep::rows_tiles(t, N);
    return U < t.ctas ? U : t.ctas;
}

// Kinds whose blocks wait on one another (the stream-K fix-up, the K-piece
// reducer, the wide reduce-scatter) need every block of a launch resident at
// once: a block that waits on one still queued behind it would only give up.
// False when the launch's grid exceeds the blocks the device holds together.
bool grid_resident(const dep_tactic_t &t, int64_t N, int64_t K, int sm_count)
{
    int64_t grid = 0;
    int per_sm = 0;
    switch (t.kind) {
    case DEP_KIND_TC:
        grid = std::min<int64_t>(t.ctas, dep::tc_units(t, N, K));
        per_sm = dep::tc_blocks_per_sm(t);
        break;
    case DEP_KIND_TC_SPLIT:
        grid = std::min<int64_t>(t.ctas, dep::tcs_items(t, N, K));
        per_sm = dep::tcs_blocks_per_sm(t);
        break;
    case DEP_KIND_TC_WIDE:
        grid = std::min<int64_t>(t.ctas, dep::wide_units(t, N, K));
        per_sm = dep::wide_blocks_per_sm(t);
        break;
    default: return true;  // no waits between blocks, or (clusters) waits only inside a co-scheduled cluster
    }
    return grid <= (int64_t)per_sm * sm_count;
}

// Split-K partial floats a launch of tactic t on an [N,K] weight may write.
size_t tactic_ws_floats(const dep_tactic_t &t, int64_t N, int64_t K)
{
    if (t.kind == DEP_KIND_TC_SPLIT)
        return 0;
    return (size_t)effective_ctas(t, N, K) * ws_per_cta(t);
}

// Exchange words a launch of tactic t may use (tensor-core kinds).
size_t tactic_xch_words(const dep_tactic_t &t, int64_t N, int64_t K)
{
    return t.kind == DEP_KIND_TC_SPLIT ? dep::tcs_xch_words(t, N, K)
           : t.kind == DEP_KIND_TC     ? dep::tc_xch_words(t, N, K)
                                       : 0;
}

size_t tactic_counters(const dep_tactic_t &t, int64_t N, int64_t K)
{
    switch (t.kind) {
    case DEP_KIND_SPLITK_FMA: return dep::fma_counters(t, N);
    case DEP_KIND_TC: return 0;  // the exchange words need no counters
    case DEP_KIND_TC_WIDE: return (size_t)effective_ctas(t, N, K) * dep::wide_flags_per_cta(t);  // flags
    case DEP_KIND_TC_CLUSTER: return 0;  // partials stay in the cluster's shared memory
    case DEP_KIND_TC_XM: return 0;       // whole K per block: no partials, no counters
    case DEP_KIND_WARP_MMA: return 0;    // whole K per block
    case DEP_KIND_TC_SPLIT: return dep::tcs_counters(t, N);
    default: return 2;  // tile dispenser and finish count (the last two counters)
    }
}

dep_tactic_t fma_tactic(int32_t rows, int32_t cols, int32_t stages, int sm_count, bool host_only,
                        int32_t tile_n = 32)
{
    dep_tactic_t t{};
    t.max_rows = rows;
    t.kind = DEP_KIND_SPLITK_FMA;
    t.tile_k = 256;
    t.cols = cols;
    t.tile_n = tile_n;
    t.stages = stages;
    int per_sm = host_only ? 1 : dep::fma_blocks_per_sm(t);
    t.ctas = sm_count * (per_sm < 1 ? 1 : per_sm);
    return t;
}

dep_tactic_t rows_tactic(int32_t rows, int32_t cols, int32_t tile_n, int32_t tile_k, int32_t stages, int32_t ctas)
{
    dep_tactic_t t{};
    t.max_rows = rows;
    t.kind = DEP_KIND_ROWS;
    t.cols = cols;
    t.tile_n = tile_n;
    t.tile_k = tile_k;
    t.stages = stages;
    t.ctas = ctas;
    return t;
}

dep_tactic_t tc_tactic(int32_t rows, int32_t cols, int32_t stages, int32_t ctas, int32_t tile_k = 64)
{
    dep_tactic_t t{};
    t.max_rows = rows;
    t.kind = DEP_KIND_TC;
    t.tile_n = 128;
    t.tile_k = tile_k;
    t.cols = cols;
    t.stages = stages;
    t.ctas = ctas;
    return t;
}

dep_tactic_t tcs_tactic(int32_t rows, int32_t cols, int32_t stages, int32_t ctas, int32_t tile_k, int32_t splits,
                        int32_t tile_n)
{
    dep_tactic_t t = tc_tactic(rows, cols, stages, ctas, tile_k);
    t.kind = DEP_KIND_TC_SPLIT;
    t.tile_n = tile_n;
    t.splits = splits;
    return t;
}

dep_tactic_t wide_tactic(int32_t rows, int32_t cols, int32_t groups_of_tiles, int32_t stages, int32_t ctas,
                         int32_t tile_k = 64)
{
    dep_tactic_t t = tc_tactic(rows, cols, stages, ctas, tile_k);
    t.kind = DEP_KIND_TC_WIDE;
    t.tile_n = 128 * groups_of_tiles;
    return t;
}

dep_tactic_t cluster_tactic(int32_t rows, int32_t cols, int32_t groups_of_tiles, int32_t k, int32_t stages,
                            int32_t ctas)
{
    dep_tactic_t t = tc_tactic(rows, cols, stages, ctas, 64);
    t.kind = DEP_KIND_TC_CLUSTER;
    t.tile_n = 128 * groups_of_tiles;
    t.splits = k;
    return t;
}

dep_tactic_t xm_tactic(int32_t rows, int32_t cols, int32_t tile_n, int32_t tile_k, int32_t stages, int32_t ctas)
{
    dep_tactic_t t = tc_tactic(rows, cols, stages, ctas, tile_k);
    t.kind = DEP_KIND_TC_XM;
    t.tile_n = tile_n;
    return t;
}

// Weight rows per tile of the x-on-M kind: the smallest multiple of 16 that
// deals the rows out in as few waves of the SMs as tiles of at most 128 rows
// allow (128 keeps two accumulator buffers in TMEM).  DSA 14560: 96 (152
// tiles); KDA 49376: 112 (441 tiles, three waves); o_proj 7168: 48 (150).
int32_t xm_rows_per_tile(int64_t N, int sm_count)
{
    const int64_t waves = std::max<int64_t>(1, (N + 128 * (int64_t)sm_count - 1) / (128 * (int64_t)sm_count));
    const int64_t per = (N + waves * sm_count - 1) / (waves * sm_count);
    return (int32_t)std::max<int64_t>(16, (per + 15) / 16 * 16);
}

dep_tactic_t mma_rows_tactic(int32_t rows, int32_t tile_k, int32_t stages)
{
    dep_tactic_t t{};
    t.max_rows = rows;
    t.kind = DEP_KIND_WARP_MMA;
    t.ctas = 1;  // one block per 16-row tile whatever this says
    t.tile_n = 16;
    t.tile_k = tile_k;
    t.stages = stages;
    t.cols = 16;
    return t;
}

// Weight rows per tile of the x-on-M kind in pairs of blocks (a cluster of two,
// each half of K): the smallest multiple of 32 that deals the rows out to the
// SMs / 2 pairs in as few waves as tiles of at most 256 rows allow.  DSA 14560:
// 192 (76 tiles); o_proj 7168: 96 (75); KDA 49376: 224 (221 tiles, three waves).
int32_t xm_pair_rows_per_tile(int64_t N, int sm_count)
{
    const int64_t pairs = std::max(1, sm_count / 2);
    const int64_t waves = std::max<int64_t>(1, (N + 256 * pairs - 1) / (256 * pairs));
    const int64_t per = (N + waves * pairs - 1) / (waves * pairs);
    return (int32_t)std::max<int64_t>(32, (per + 31) / 32 * 32);
}

// Deepest pipeline of the tensor-core kernel that fits in shared memory.
int32_t tc_default_stages(int32_t cols)
{
    for (int32_t st : {8, 6, 4, 3, 2})
        if (dep::tc_valid(tc_tactic(1, cols, st, 1)))
            return st;
    return 2;
}

// The fixed rule (runtime.hybrid page, HybridAttention.__init__: warp split-K
// for the smallest batches, the GEMM path past them; the split point moves to
// where each kernel measured fastest on this GPU):
//  * one or two x rows: whole weight rows on the FMA pipe (no cross-block split);
//  * up to 16 rows (a 16-wide MMA): the tensor cores over fixed K pieces taken
//    dynamically -- SMs / tiles pieces per 128-row tile while the tiles fit on
//    the SMs (o_proj: 2, DSA: 1, one item per block), 3 pieces otherwise (KDA:
//    386 tiles, 1158 items);
//  * 32 rows, and wider batches the rule below does not give to clusters: the
//    stream-K tensor-core kernel, one block per tile when the tiles nearly fill
//    the GPU;
//  * 64 rows and more: a thread-block cluster per group of weight tiles (below).
// Measured on GB300 (per call, CUDA events): at 4 rows the K-piece tensor-core
// tactic is 1.9-2.8 us faster than the stream-K FMA kernel and 3-34 us faster
// than the whole-row kernel on all three weights; at 4-16 rows it is 0.2-1.5 us
// faster than the stream-K tensor-core kernel for o_proj, equal for DSA and up
// to 1 us faster for KDA.
dep_tactic_t default_tactic(int32_t rows, int64_t N, int64_t K, int sm_count)
{
    if (rows <= 2) {
        // Whole rows, no cross-block split: 16-row tiles, stages of 1024
        // columns, handed out dynamically (measured on GB300: 5-8 % faster than
        // the stream-K FMA kernel at one x row, on all three weights).  One x
        // row takes six stages (per call, CUDA graph + PDL: o_proj / DSA / KDA
        // 25.6 / 29.8 / 94.7 us against 26.0 / 30.0 / 95.0 at four), two rows
        // four (DSA: 32.6 against 32.9 at six; o_proj: six do not fit beside
        // x).  Falls through where x does not fit in shared memory.
        const int32_t cols = pow2_at_least(rows);
        for (int32_t st : {rows == 1 ? 6 : 4, 4}) {
            const dep_tactic_t t = rows_tactic(rows, cols, 16, 1024, st, sm_count);
            if (dep::rows_fits(t, K))
                return t;
        }
    }
    const int32_t cols = std::min<int32_t>(256, std::max<int32_t>(16, pow2_at_least(rows)));
    const int64_t tiles = (N + 127) / 128, t64 = (N + 63) / 64;
    // 17 to 256 batch rows: x on the MMA's M side (tc_xm.cu) against tiles of
    // R weight rows that fill the SMs, where the x bytes of a 64-column step are
    // at most 1.5x the weight's (x rows padded to 64, 128 or 256): whole K per
    // block where R allows that, else a pair of blocks (a cluster of two, each
    // half of K) per tile of up to twice the rows.  Stages of the widest slice
    // count that still gives a ring of three beside x of the pass's height, the
    // deepest ring that fits.  Measured on GB300 per call (CUDA graph + PDL,
    // weights past L2): DSA 14560 x 7168 B = 32 / 64 / 128: 32.4 / 32.6 / 33.4 us
    // against 33.1 / 35.9 / 39.7 us for the stream-K and cluster kinds, B = 256
    // (pairs, R = 192): 41.3 against 45.8 us; KDA 49376 x 7168 B = 64 / 128:
    // 100.8 / 107.6 against 108.4 / 112.5 us, B = 256 (pairs, R = 224): 142.8
    // against 147.7 us; o_proj 7168 x 12288 B = 32 / 64: 28.8 / 28.8 against
    // 29.5 / 33.1 us, B = 128 (pairs, R = 96): 32.4 against 37.1 us.  o_proj at
    // 256 rows keeps the cluster kind (x's bytes would be 2.7x the weight's).
    if (rows > 16 && rows <= 256) {
        const int32_t xrows = rows <= 64 ? 64 : (rows <= 128 ? 128 : 256);
        const int32_t xcols = rows <= 128 ? 128 : 256;  // one or two blocks of 128 rows per pass
        const int32_t xr = rows <= 64 ? 64 : 128;       // x rows per block of a pass
        auto pick = [&](int32_t R, int32_t splits, int32_t ctas) {
            dep_tactic_t none{};
            if (R > 256 || 2 * xrows > 3 * R)
                return none;
            for (int32_t tk : {256, 128, 64})
                if (dep::xm_stages_fit(R, tk, xcols, xr) >= 3) {
                    dep_tactic_t t = xm_tactic(rows, xcols, R, tk, dep::xm_stages_fit(R, tk, xcols, 128), ctas);
                    t.splits = splits;
                    if (dep::xm_valid(t))
                        return t;
                }
            return none;
        };
        dep_tactic_t t = pick(xm_rows_per_tile(N, sm_count), 0, sm_count);
        if (t.kind == 0) {
            const int32_t R2 = xm_pair_rows_per_tile(N, sm_count);
            const int64_t pairs = std::min<int64_t>((N + R2 - 1) / R2, sm_count / 2);
            t = pick(R2, 2, (int32_t)(2 * pairs));
        }
        if (t.kind != 0)
            return t;
    }
    // 6 to 16 rows where tiles of 16 weight rows number 2.5 to 4 per SM (o_proj
    // 7168 rows and its TP shards, the TP-2 DSA shard: 448-455 tiles on 152
    // SMs): the warp-level MMA kind, which holds no tensor memory, so three of
    // its blocks share an SM and the next call's blocks stream beside the
    // current call's.  Measured on GB300 per call (CUDA graph + PDL, weights
    // past L2), B = 16: o_proj 27.7 against 28.5 us for 64-row K-piece tiles;
    // the 8-layer chain as one graph 489.5 against 496.8 us; TP shards o_proj
    // K = 6144 / 3072 / 1536: 15.0 / 8.8 / 5.3 against 16.3 / 9.8 / 5.9 us, DSA
    // 7280 rows 17.2 against 18.6 us.  Slower with fewer tiles per SM (3640 DSA
    // rows: 13.9 against 11.6 us), with more (14560: 33.6 against 32.7 us), and
    // at up to 4 rows (o_proj B = 4: 33.1 against 28.3 us).
    if (rows >= 6 && rows <= 16) {
        const int64_t t16 = (N + 15) / 16;
        if (2 * t16 >= 5 * (int64_t)sm_count && t16 <= 4 * (int64_t)sm_count) {
            const dep_tactic_t t = mma_rows_tactic(rows, 256, K <= 2048 ? 3 : 4);
            if (dep::mma_rows_valid(t))
                return t;
        }
    }
    // Up to 32 batch rows on long weight rows (K >= 3072) whose 64-row tiles fit
    // on the SMs: 64-row K-piece tiles in as few pieces as fill the SMs (o_proj:
    // 112 tiles, one piece each, no exchange).  Measured on GB300 per call (CUDA
    // graph + PDL, weights rotated past L2), o_proj 7168 x 12288: B = 32 29.9 us
    // against 33.4 us for the stream-K kernel; B = 4 / 16 28.4 / 28.6 us against
    // 28.7 / 29.2 us for 128-row tiles in two pieces.  On shorter rows 128-row
    // tiles in pieces win (7168 x 1536: 5.9 against 6.3 us): three 64 KB stages
    // hold a whole 196 KB item before the wait for x, five 32 KB stages do not.
    if (cols <= 32 && t64 <= sm_count && K >= 3072) {
        const int32_t splits = (int32_t)std::min<int64_t>(64, std::max<int64_t>(1, sm_count / t64));
        for (int32_t st : {6, 5, 4, 3}) {
            const dep_tactic_t t = tcs_tactic(rows, cols, st, sm_count, 256, splits, 64);
            if (dep::tcs_valid(t))
                return t;
        }
    }
    // Widest stage (most contiguous bytes per weight row) that still leaves a
    // ring of at least three stages.
    if (cols == 16) {
        const int32_t splits =
            tiles <= sm_count ? (int32_t)std::min<int64_t>(64, std::max<int64_t>(1, sm_count / tiles)) : 3;
        for (int32_t tk : {256, 128})
            for (int32_t st : {6, 5, 4, 3}) {
                const dep_tactic_t t = tcs_tactic(rows, cols, st, sm_count, tk, splits, 128);
                if (dep::tcs_valid(t))
                    return t;
            }
    }
    // 64 batch rows and more: a cluster of k CTAs per group of two 128-row
    // tiles (x bytes per weight byte halved; the K pieces added through
    // distributed shared memory), k = SMs / groups up to 4, while the groups fit
    // on the SMs in one wave of clusters of two; at 256 rows also past that.
    // Where they do not, 128 rows take groups of four tiles, one CTA each, if
    // those fit.  Measured on GB300 (per launch, back to back): DSA 14560 x
    // 7168 B = 128 / 256: 44.6 / 50.0 us against 45.4 / 61.0 us for the one-tile
    // kernel; o_proj 7168 x 12288 B = 64..256 (k = 4): 37.2 / 41.0 / 49.9 us; KDA
    // 49376 x 7168 B = 128 (four-tile groups) / 256 (k = 2): 119.6 / 152.6 us.
    // At 64 rows on a weight whose 128-row tiles nearly fill the SMs (DSA: 114
    // tiles), one tile per block of the stream-K kernel, no K split, measured
    // faster than clusters of two (36.6 against 38.1 us per call, CUDA graph + PDL).
    const bool one_tile_each = tiles <= sm_count && 4 * tiles >= 3 * (int64_t)sm_count;
    if (cols >= 64 && !(cols == 64 && one_tile_each)) {
        const int64_t t2 = (N + 255) / 256, t3 = (N + 191) / 192, t4 = (N + 511) / 512;
        const int32_t sw = cols == 256 ? 4 : (cols == 128 ? 6 : 5);
        if (cols == 256 && 2 * t3 <= sm_count && 8 * t3 > 3 * (int64_t)sm_count) {
            // 256 rows: groups of 192 rows (a 128-row and a 64-row tile) in clusters
            // of two where those nearly fill the SMs (DSA: 76 groups, 152 CTAs;
            // 49.4 us against 50.6 us for 57 groups of two tiles on 114 CTAs)
            dep_tactic_t t = cluster_tactic(rows, cols, 2, 2, 5, (int32_t)t3 * 2);
            t.tile_n = 192;
            if (dep::cluster_valid(t))
                return t;
        }
        if (2 * t2 <= sm_count) {
            const int32_t k = (int32_t)std::min<int64_t>(4, sm_count / t2);
            const dep_tactic_t t = cluster_tactic(rows, cols, 2, k, sw, (int32_t)t2 * k);
            if (dep::cluster_valid(t))
                return t;
        } else if (cols == 256) {
            const dep_tactic_t t = cluster_tactic(rows, cols, 2, 2, sw, (sm_count / 2) * 2);
            if (dep::cluster_valid(t))
                return t;
        } else if (cols == 128 && t4 <= sm_count) {
            const dep_tactic_t t = cluster_tactic(rows, cols, 4, 1, 3, (int32_t)t4);
            if (dep::cluster_valid(t))
                return t;
        }
    }
    const int32_t ctas = one_tile_each ? (int32_t)tiles : sm_count;
    // 64-column stages for the widest batches.
    for (int32_t tk : {256, 128}) {
        for (int32_t st : {6, 5, 4, 3}) {
            const dep_tactic_t t = tc_tactic(rows, cols, st, ctas, tk);
            if (dep::tc_valid(t))
                return t;
        }
    }
    return tc_tactic(rows, cols, tc_default_stages(cols), ctas);
}

void sort_table(std::vector<dep_tactic_t> &table)
{
    std::sort(table.begin(), table.end(),
              [](const dep_tactic_t &a, const dep_tactic_t &b) { return a.max_rows < b.max_rows; });
}

const dep_tactic_t *lookup(const dep_plan_s *p, int32_t B)
{
    std::vector<int32_t> keys;
    keys.reserve(p->table.size());
    for (const auto &t : p->table)
        keys.push_back(t.max_rows);
    const int32_t i = dep_bins_index(keys.data(), (int32_t)keys.size(), B);
    return i < 0 ? nullptr : &p->table[(size_t)i];
}

// Allocate (or re-allocate) the plan's device block for its current table.
dep_status_t allocate_device(dep_plan_s *p, size_t extra_ws_floats = 0, size_t extra_counters = 0,
                             size_t extra_xch_words = 0)
{
    // Room for the table's tactics, for any tactic of the same per-block
    // footprint on up to one block per SM, and for FMA-sized footprints on up to
    // four blocks per SM (explicit tactics of tests and tuning use other grids).
    size_t ws = std::max(extra_ws_floats, (size_t)4 * (size_t)p->sm_count * 512);
    size_t cnt = std::max<size_t>(256, extra_counters);
    size_t xw = extra_xch_words;
    int32_t rows = 1;
    for (const auto &t : p->table) {
        ws = std::max(ws, tactic_ws_floats(t, p->N, p->K));
        ws = std::max(ws, (size_t)p->sm_count * ws_per_cta(t));
        cnt = std::max(cnt, tactic_counters(t, p->N, p->K));
        xw = std::max(xw, tactic_xch_words(t, p->N, p->K));
        // Room for the stream-K tensor-core kernels on every SM at this width
        // (explicit tactics of tests and tuning), whatever kind the table holds.
        if (t.kind == DEP_KIND_TC || t.kind == DEP_KIND_TC_SPLIT || t.kind == DEP_KIND_TC_WIDE ||
            t.kind == DEP_KIND_TC_CLUSTER) {
            dep_tactic_t one = t;
            one.tile_n = 128;
            xw = std::max(xw, (size_t)p->sm_count * dep::tc_xch_words_per_cta(one));
        }
        if (t.kind == DEP_KIND_TC_WIDE)
            cnt = std::max(cnt, (size_t)p->sm_count * dep::wide_flags_per_cta(t));
        rows = std::max(rows, t.max_rows);
    }
    auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
    const size_t status_b = 256, cnt_b = up(cnt * sizeof(int)), xch_b = up(xw * 8), ws_b = up(ws * sizeof(float));
    const size_t xs_b = up((size_t)rows * p->K * 2), ys_b = up((size_t)rows * p->N * 2);
    const size_t total = status_b + cnt_b + xch_b + ws_b + xs_b + ys_b;
    if (p->dev_block && cnt <= p->n_counters && xw <= p->xch_words && ws <= p->ws_floats && rows <= p->stage_rows)
        return DEP_OK;  // the current block already has room for every part
    if (env_is("DEP_FAULT", "alloc"))
        return DEP_ERR_OOM;
    void *blk = nullptr;
    if (cudaMalloc(&blk, total) != cudaSuccess) {
        cudaGetLastError();
        return DEP_ERR_OOM;
    }
    if (cudaMemset(blk, 0, status_b + cnt_b + xch_b) != cudaSuccess) {  // status, counters, exchange flags
        cudaFree(blk);
        return DEP_ERR_CUDA;
    }
    if (p->dev_block) {
        cudaDeviceSynchronize();
        cudaFree(p->dev_block);
    }
    char *c = static_cast<char *>(blk);
    p->dev_block = blk;
    p->dev_bytes = total;
    p->status = reinterpret_cast<int *>(c);
    p->counters = reinterpret_cast<int *>(c + status_b);
    p->n_counters = cnt_b / sizeof(int);
    p->xch = reinterpret_cast<unsigned long long *>(c + status_b + cnt_b);
    p->xch_words = xch_b / 8;
    p->ws = reinterpret_cast<float *>(c + status_b + cnt_b + xch_b);
    p->ws_floats = ws_b / sizeof(float);
    p->x_stage = reinterpret_cast<uint16_t *>(c + status_b + cnt_b + xch_b + ws_b);
    p->y_stage = reinterpret_cast<uint16_t *>(c + status_b + cnt_b + xch_b + ws_b + xs_b);
    p->stage_rows = rows;
    return DEP_OK;
}

dep_status_t check_shape(int64_t N, int64_t K)
{
    if (N < 1 || K < 8 || N > INT32_MAX || K > INT32_MAX)
        return K > 0 && K < 8 && K % 8 ? DEP_ERR_MISALIGNED : DEP_ERR_INVALID_ARG;
    if (K % 8)
        return DEP_ERR_MISALIGNED;
    return DEP_OK;
}

dep_status_t make_plan(int64_t N, int64_t K, const int32_t *batches, int32_t n_batches,
                       bool host_only, int32_t sm_count, dep_plan_t *out)
{
    if (!out)
        return DEP_ERR_INVALID_ARG;
    *out = nullptr;
    dep_status_t st = check_shape(N, K);
    if (st != DEP_OK)
        return st;
    if (n_batches < 0 || (n_batches > 0 && !batches))
        return DEP_ERR_INVALID_ARG;
    std::vector<int32_t> bs;
    if (n_batches == 0)
        bs.assign(std::begin(kDefaultBatches), std::end(kDefaultBatches));
    else
        bs.assign(batches, batches + n_batches);
    for (int32_t b : bs)
        if (b < 1)
            return DEP_ERR_INVALID_ARG;
    std::sort(bs.begin(), bs.end());
    bs.erase(std::unique(bs.begin(), bs.end()), bs.end());

    dep_plan_s *p = new (std::nothrow) dep_plan_s;
    if (!p)
        return DEP_ERR_OOM;
    p->N = N;
    p->K = K;
    p->host_only = host_only;
    p->log = env_is("DEP_LOG", "1");
    p->fault_launch = env_is("DEP_FAULT", "launch");
    if (host_only) {
        if (sm_count < 1) {
            delete p;
            return DEP_ERR_INVALID_ARG;
        }
        p->sm_count = sm_count;
        p->device_name = "host";
    } else {
        cudaDeviceProp prop;
        if (cudaGetDevice(&p->device) != cudaSuccess ||
            cudaGetDeviceProperties(&prop, p->device) != cudaSuccess) {
            cudaGetLastError();
            delete p;
            return DEP_ERR_CUDA;
        }
        p->sm_count = prop.multiProcessorCount;
        p->device_name = prop.name;
        if (prop.major * 10 + prop.minor < 100) {
            delete p;
            return DEP_ERR_UNSUPPORTED;
        }
        if (dep::fma_prepare_device() != cudaSuccess || dep::tc_prepare_device() != cudaSuccess ||
            dep::tcs_prepare_device() != cudaSuccess || dep::wide_prepare_device() != cudaSuccess ||
            dep::cluster_prepare_device() != cudaSuccess || dep::xm_prepare_device() != cudaSuccess ||
            dep::mma_rows_prepare_device() != cudaSuccess ||
            dep::rows_prepare_device() != cudaSuccess) {
            cudaGetLastError();
            delete p;
            return DEP_ERR_CUDA;
        }
    }
    for (int32_t b : bs)
        p->table.push_back(default_tactic(b, N, K, p->sm_count));
    sort_table(p->table);
    if (!host_only) {
        st = allocate_device(p);
        if (st != DEP_OK) {
            delete p;
            return st;
        }
    }
    if (p->log)
        for (const auto &t : p->table)
            std::fprintf(stderr, "[dep] N=%lld K=%lld rows<=%d kind=%d ctas=%d tile_n=%d stages=%d cols=%d\n",
                         (long long)N, (long long)K, t.max_rows, t.kind, t.ctas, t.tile_n, t.stages, t.cols);
    *out = p;
    return DEP_OK;
}

dep_status_t run_impl(dep_plan_t p, const dep_tactic_t *t, const void *x, const void *W, void *y,
                      int32_t B, void *stream,
                      bool force_pdl = false)
{
    if (!p || B < 0)
        return DEP_ERR_INVALID_ARG;
    if (p->host_only)
        return DEP_ERR_UNSUPPORTED;
    if (B == 0)
        return DEP_OK;
    if (!x || !W || !y || !t)
        return DEP_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(W) || !aligned16(y))
        return DEP_ERR_MISALIGNED;
    const size_t xb = (size_t)B * p->K * 2, wb = (size_t)p->N * p->K * 2, yb = (size_t)B * p->N * 2;
    if (overlaps(y, yb, x, xb) || overlaps(y, yb, W, wb))
        return DEP_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != p->device) {
        cudaGetLastError();
        return DEP_ERR_INVALID_ARG;
    }
    if (tactic_ws_floats(*t, p->N, p->K) > p->ws_floats || tactic_counters(*t, p->N, p->K) > p->n_counters ||
        tactic_xch_words(*t, p->N, p->K) > p->xch_words)
        return DEP_ERR_INVALID_ARG;
    if (p->fault_launch)
        return DEP_ERR_CUDA;
    RunArgs a;
    a.x = static_cast<const uint16_t *>(x);
    a.W = static_cast<const uint16_t *>(W);
    a.y = static_cast<uint16_t *>(y);
    a.B = B;
    a.N = p->N;
    a.K = p->K;
    a.ws = p->ws;
    a.ws_floats = p->ws_floats;
    a.counters = p->counters;
    a.n_counters = p->n_counters;
    a.xch = p->xch;
    a.xch_words = p->xch_words;
    a.status = p->status;
    a.stream = static_cast<cudaStream_t>(stream);
    a.wait_limit_ns = p->wait_limit_ns;
    a.pdl = p->pdl || force_pdl;
    a.keep_pieces = p->keep_pieces;
    if (t->kind == DEP_KIND_ROWS && !dep::rows_fits(*t, p->K))
        return DEP_ERR_UNSUPPORTED;  // x and the ring do not fit in shared memory for this K
    cudaError_t e = t->kind == DEP_KIND_SPLITK_FMA ? dep::fma_run(*t, a)
                    : t->kind == DEP_KIND_TC       ? dep::tc_run(*t, a)
                    : t->kind == DEP_KIND_TC_SPLIT ? dep::tcs_run(*t, a)
                    : t->kind == DEP_KIND_TC_WIDE  ? dep::wide_run(*t, a)
                    : t->kind == DEP_KIND_TC_CLUSTER ? dep::cluster_run(*t, a)
                    : t->kind == DEP_KIND_TC_XM    ? dep::xm_run(*t, a)
                    : t->kind == DEP_KIND_WARP_MMA ? dep::mma_rows_run(*t, a)
                                                   : dep::rows_run(*t, a);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return DEP_ERR_CUDA;
    }
    return DEP_OK;
}

// ---- tuning (DEP_PLAN_TUNE) ----

__global__ void fill_bf16_kernel(uint16_t *p, size_t n, uint64_t seed)
{
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        uint64_t z = seed + 0x9E3779B97F4A7C15ull * (i + 1);
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        z ^= z >> 31;
        // random sign and fraction, magnitude in [2^-8, 2): ordinary finite values
        p[i] = (uint16_t)(((z >> 16) & 0x8000u) | ((119u + (uint32_t)(z % 9u)) << 7) | ((z >> 32) & 0x7Fu));
    }
}

std::vector<dep_tactic_t> candidates(int32_t rows, int64_t N, int64_t K, int sm_count)
{
    std::vector<dep_tactic_t> c;
    if (rows <= 8) {
        const int32_t cols = pow2_at_least(rows);
        for (int32_t tn : {32, 64})
            for (int32_t st : {4, 6, 8})
                c.push_back(fma_tactic(rows, cols, st, sm_count, false, tn));
    }
    if (rows <= 4) {
        const int32_t cols = pow2_at_least(rows);
        for (int32_t tn : {8, 16})
            for (int32_t kc : {1024, 2048, 4096})
                for (int32_t st : {2, 3, 4, 6})
                    c.push_back(rows_tactic(rows, cols, tn, kc, st, sm_count));
    }
    const int32_t cols = std::min<int32_t>(256, std::max<int32_t>(16, pow2_at_least(rows)));
    const int64_t tiles = (N + 127) / 128;
    // Grids: every SM (stream-K), and for weights with fewer 128-row tiles than
    // SMs also one, two and four blocks per tile (less splitting, fewer partials).
    std::vector<int32_t> grids{sm_count};
    for (int64_t per : {1, 2, 4})
        if (per * tiles < sm_count)
            grids.push_back((int32_t)(per * tiles));
    for (int32_t tk : {64, 128, 256})
        for (int32_t st : {2, 3, 4, 6, 8, 10, 12})
            for (int32_t g : grids)
                c.push_back(tc_tactic(rows, cols, st, g, tk));
    // Fixed K pieces taken dynamically, on 64- and 128-row tiles: 1 to 8
    // pieces per tile, and as many as give about one item per SM.
    for (int32_t bm : {64, 128}) {
        const int64_t t_bm = (N + bm - 1) / bm;
        std::vector<int32_t> pieces{1, 2, 3, 4, 8};
        const int32_t fill = (int32_t)std::min<int64_t>(64, std::max<int64_t>(1, sm_count / t_bm));
        if (std::find(pieces.begin(), pieces.end(), fill) == pieces.end())
            pieces.push_back(fill);
        for (int32_t tk : {128, 256})
            for (int32_t st : {3, 4, 5, 6})
                for (int32_t sp : pieces)
                    c.push_back(tcs_tactic(rows, cols, st, sm_count, tk, sp, bm));
    }
    // Groups of 2 or 4 weight tiles per x slice (wide batches), stream-K on every SM.
    if (cols >= 32)
        for (int32_t g : {2, 4})
            for (int32_t tk : {64, 128})
                for (int32_t st : {2, 3, 4, 5, 6})
                    if (cols * g <= 512)
                        c.push_back(wide_tactic(rows, cols, g, st, sm_count, tk));
    // A cluster of k CTAs per group of 2 or 4 tiles (or a 128-row and a 64-row
    // tile, 192 rows): k = 1..4, as many clusters as groups (at most one wave of
    // the SMs).
    if (cols >= 32)
        for (int32_t grows : {256, 192, 512})
            for (int32_t k : {1, 2, 3, 4})
                for (int32_t st : {3, 4, 5, 6}) {
                    if (cols * (grows == 192 ? 2 : grows / 128) > 512 || (grows == 192 && cols < 64))
                        continue;
                    const int64_t groups = (N + grows - 1) / grows;
                    const int32_t clusters = (int32_t)std::max<int64_t>(1, std::min<int64_t>(groups, sm_count / k));
                    dep_tactic_t t = cluster_tactic(rows, cols, 2, k, st, clusters * k);
                    t.tile_n = grows;
                    c.push_back(t);
                }
    // x on the MMA's M side: tiles of 16..256 weight rows (the default's R and
    // its neighbours, and the multiples of 16 that fill the SMs in one, two or
    // three waves), two or four slices per stage, every depth that fits.
    if (rows > 16) {
        const int32_t xcols = rows <= 128 ? 128 : 256;
        std::vector<int32_t> rs;
        const int32_t r0 = xm_rows_per_tile(N, sm_count);
        for (int32_t r : {r0 - 16, r0, r0 + 16, r0 + 32})
            rs.push_back(r);
        for (int64_t w : {1, 2, 3}) {
            const int64_t per = (N + w * sm_count - 1) / (w * sm_count);
            rs.push_back((int32_t)((per + 15) / 16 * 16));
        }
        std::sort(rs.begin(), rs.end());
        rs.erase(std::unique(rs.begin(), rs.end()), rs.end());
        for (int32_t r : rs)
            for (int32_t tk : {128, 256})
                for (int32_t st : {2, 3, 4, 5, 6})
                    if (r >= 16 && r <= 256)
                        c.push_back(xm_tactic(rows, xcols, r, tk, st, sm_count));
        // pairs of blocks per tile (each half of K)
        const int32_t p0 = xm_pair_rows_per_tile(N, sm_count);
        for (int32_t r : {p0 - 32, p0, p0 + 32}) {
            if (r < 32 || r > 256)
                continue;
            const int64_t pairs = std::min<int64_t>((N + r - 1) / r, sm_count / 2);
            for (int32_t tk : {64, 128})
                for (int32_t st : {2, 3, 4, 5, 6}) {
                    dep_tactic_t t = xm_tactic(rows, xcols, r, tk, st, (int32_t)(2 * pairs));
                    t.splits = 2;
                    c.push_back(t);
                }
        }
    }
    // Warp-level MMAs on 16-row tiles (no tensor memory), up to 16 rows: whole
    // K per block, or two K pieces per tile in a cluster.
    if (rows <= 16)
        for (int32_t sp : {0, 2})
            for (int32_t tk : {128, 256})
                for (int32_t st : {3, 4, 6}) {
                    dep_tactic_t t = mma_rows_tactic(rows, tk, st);
                    t.splits = sp;
                    c.push_back(t);
                }
    // K pieces keep every piece's partial: leave out tactics whose exchange words
    // would take more than 64 MB.
    constexpr size_t kMaxPieceWords = (64u << 20) / 8;
    std::vector<dep_tactic_t> ok;
    for (const auto &t : c)
        if (tactic_valid(t) && (t.kind != DEP_KIND_ROWS || dep::rows_fits(t, K)) &&
            (t.kind != DEP_KIND_TC_SPLIT || tactic_xch_words(t, N, K) <= kMaxPieceWords))
            ok.push_back(t);
    return ok;
}

// Time every candidate of every table entry on scratch data of the plan's shape
// (enough distinct weight copies that no launch reads its weight from L2) and
// keep the fastest.  Median of timed launches, CUDA events on a private stream.
dep_status_t tune_plan(dep_plan_s *p)
{
    std::vector<std::vector<dep_tactic_t>> cands;
    size_t ws_need = 0, cnt_need = 0, xch_need = 0;
    int32_t rows_max = 1;
    for (const auto &t : p->table) {
        cands.push_back(candidates(t.max_rows, p->N, p->K, p->sm_count));
        for (const auto &c : cands.back()) {
            ws_need = std::max(ws_need, tactic_ws_floats(c, p->N, p->K));
            cnt_need = std::max(cnt_need, tactic_counters(c, p->N, p->K));
            xch_need = std::max(xch_need, tactic_xch_words(c, p->N, p->K));
        }
        rows_max = std::max(rows_max, t.max_rows);
    }
    dep_status_t st = allocate_device(p, ws_need, cnt_need, xch_need);
    if (st != DEP_OK)
        return st;
    int l2 = 0;
    cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, p->device);
    const size_t wbytes = (size_t)p->N * p->K * 2;
    size_t copies = std::max<size_t>(2, (2 * (size_t)l2 + wbytes - 1) / wbytes);
    copies = std::min<size_t>(copies, 64);
    const size_t xbytes = (size_t)rows_max * p->K * 2, ybytes = (size_t)rows_max * p->N * 2;
    char *scratch = nullptr;
    if (cudaMalloc(&scratch, copies * wbytes + xbytes + ybytes + 512) != cudaSuccess) {
        cudaGetLastError();
        return DEP_ERR_OOM;
    }
    uint16_t *Wc = reinterpret_cast<uint16_t *>(scratch);
    uint16_t *xs = reinterpret_cast<uint16_t *>(scratch + ((copies * wbytes + 255) & ~(size_t)255));
    uint16_t *ys = reinterpret_cast<uint16_t *>(reinterpret_cast<char *>(xs) + ((xbytes + 255) & ~(size_t)255));
    cudaStream_t s = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    bool ok = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreate(&e0) == cudaSuccess && cudaEventCreate(&e1) == cudaSuccess;
    if (ok) {
        fill_bf16_kernel<<<1024, 256, 0, s>>>(Wc, copies * wbytes / 2, 12345);
        fill_bf16_kernel<<<64, 256, 0, s>>>(xs, xbytes / 2, 777);
        ok = cudaGetLastError() == cudaSuccess && cudaStreamSynchronize(s) == cudaSuccess;
    }
    size_t turn = 0;
    // Batches of 8 back-to-back launches between one pair of events (event
    // timestamps are coarse, about 2 us on GB300), the best of 3 batches after 2
    // warm-up launches.  (Timing the same 8 launches as a captured CUDA graph
    // ranked the candidates of each call alike within 0.1-0.3 us, but the
    // tables it chose ran the tensor-parallel shard step 9 % slower as one
    // graph, measured on one GB300, so the launches stay eager.)
    auto time_launches = [&](const dep_tactic_t &c, int32_t B, float &ms_out) -> bool {
        for (int w = 0; w < 2; ++w)
            if (run_impl(p, &c, xs, Wc + (turn++ % copies) * (wbytes / 2), ys, B, s) != DEP_OK)
                return false;
        float best_ms = 1e30f;
        for (int rep = 0; rep < 3; ++rep) {
            if (cudaEventRecord(e0, s) != cudaSuccess)
                return false;
            for (int l = 0; l < 8; ++l)
                if (run_impl(p, &c, xs, Wc + (turn++ % copies) * (wbytes / 2), ys, B, s) != DEP_OK)
                    return false;
            float t = 0;
            if (cudaEventRecord(e1, s) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
                cudaEventElapsedTime(&t, e0, e1) != cudaSuccess)
                return false;
            best_ms = std::min(best_ms, t / 8);
        }
        ms_out = best_ms;
        return true;
    };
    for (size_t i = 0; ok && i < p->table.size(); ++i) {
        const int32_t B = p->table[i].max_rows;
        float best = 1e30f;
        dep_tactic_t best_t = p->table[i];
        // The default rule's tactic is timed too, so that a tuned entry is never
        // slower than the default's in the tuner's own measurement.
        std::vector<dep_tactic_t> cs;
        if (tactic_valid(p->table[i]))
            cs.push_back(p->table[i]);
        cs.insert(cs.end(), cands[i].begin(), cands[i].end());
        for (const auto &c : cs) {
            float med = 0;
            ok = time_launches(c, B, med);
            if (!ok)
                break;
            if (p->log)
                std::fprintf(stderr,
                             "[dep] tune N=%lld K=%lld B=%d kind=%d cols=%d tile_n=%d tile_k=%d stages=%d ctas=%d "
                             "splits=%d: %.2f us\n",
                             (long long)p->N, (long long)p->K, B, c.kind, c.cols, c.tile_n, c.tile_k, c.stages, c.ctas,
                             c.splits, med * 1e3f);
            if (med < best) {
                best = med;
                best_t = c;
            }
        }
        best_t.max_rows = B;
        p->table[i] = best_t;
    }
    if (e0)
        cudaEventDestroy(e0);
    if (e1)
        cudaEventDestroy(e1);
    if (s) {
        cudaStreamSynchronize(s);
        cudaStreamDestroy(s);
    }
    cudaFree(scratch);
    if (!ok) {
        cudaGetLastError();
        return DEP_ERR_CUDA;
    }
    int32_t code = 0;
    if (cudaMemcpy(&code, p->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return DEP_ERR_CUDA;
    }
    return code ? DEP_ERR_TIMEOUT : DEP_OK;
}

}  // namespace

extern "C" {

int32_t dep_bins_index(const int32_t *keys, int32_t n_keys, int32_t B)
{
    if (!keys || n_keys < 1)
        return -1;
    int32_t best = -1, largest = 0;
    for (int32_t i = 0; i < n_keys; ++i) {
        if (keys[i] > keys[largest])
            largest = i;
        if (keys[i] >= B && (best < 0 || keys[i] < keys[best]))
            best = i;
    }
    return best >= 0 ? best : largest;
}

dep_status_t dep_projection_plan(int64_t N, int64_t K, const int32_t *batches, int32_t n_batches,
                                 uint32_t flags, dep_plan_t *out)
{
    if (flags & ~(DEP_PLAN_DEFAULT | DEP_PLAN_TUNE | DEP_PLAN_PDL | DEP_PLAN_KEEP_PIECES)) {
        if (out)
            *out = nullptr;
        return DEP_ERR_INVALID_ARG;
    }
    dep_status_t st = make_plan(N, K, batches, n_batches, false, 0, out);
    if (st != DEP_OK)
        return st;
    (*out)->pdl = (flags & DEP_PLAN_PDL) != 0;
    (*out)->keep_pieces = (flags & DEP_PLAN_KEEP_PIECES) != 0;
    if (!(flags & DEP_PLAN_TUNE))
        return st;
    st = tune_plan(*out);
    if (st != DEP_OK) {
        dep_projection_plan_destroy(*out);
        *out = nullptr;
    }
    return st;
}

dep_status_t dep_projection_plan_host(int64_t N, int64_t K, const int32_t *batches,
                                      int32_t n_batches, int32_t sm_count, dep_plan_t *out)
{
    return make_plan(N, K, batches, n_batches, true, sm_count, out);
}

dep_status_t dep_projection_run(dep_plan_t plan, const void *x, const void *W, void *y, int32_t B,
                                void *stream)
{
    if (!plan || B < 0)
        return DEP_ERR_INVALID_ARG;
    if (B == 0)
        return plan->host_only ? DEP_ERR_UNSUPPORTED : DEP_OK;
    return run_impl(plan, lookup(plan, B), x, W, y, B, stream);
}

dep_status_t dep_projection_run_tactic(dep_plan_t plan, const dep_tactic_t *tactic, const void *x,
                                       const void *W, void *y, int32_t B, void *stream)
{
    if (!tactic || !tactic_valid(*tactic))
        return DEP_ERR_INVALID_ARG;
    if (plan && !plan->host_only && !grid_resident(*tactic, plan->N, plan->K, plan->sm_count))
        return DEP_ERR_UNSUPPORTED;
    return run_impl(plan, tactic, x, W, y, B, stream);
}

dep_status_t dep_projection_run_host(dep_plan_t plan, const void *x_host, const void *W,
                                     void *y_host, int32_t B, void *stream)
{
    if (!plan || B < 0)
        return DEP_ERR_INVALID_ARG;
    if (plan->host_only)
        return DEP_ERR_UNSUPPORTED;
    if (B == 0)
        return DEP_OK;
    if (!x_host || !y_host || B > plan->stage_rows)
        return DEP_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t xb = (size_t)B * plan->K * 2, yb = (size_t)B * plan->N * 2;
    // Pinned (mapped) host buffers: zero-copy staging kernels chained to the
    // projection by programmatic dependent launch.  Anything else: memcpys.
    cudaPointerAttributes ax{}, ay{};
    const bool mapped = cudaPointerGetAttributes(&ax, x_host) == cudaSuccess &&
                        cudaPointerGetAttributes(&ay, y_host) == cudaSuccess && ax.type == cudaMemoryTypeHost &&
                        ay.type == cudaMemoryTypeHost && ax.devicePointer && ay.devicePointer &&
                        aligned16(ax.devicePointer) && aligned16(ay.devicePointer) && !env_is("DEP_STAGING", "copy");
    cudaGetLastError();  // the attribute query of an unregistered pointer may leave an error
    if (mapped) {
        const dep_tactic_t *t = lookup(plan, B);
        if (dep::stage_copy(static_cast<const uint16_t *>(ax.devicePointer), plan->x_stage, (size_t)B * plan->K,
                            true, s) != cudaSuccess) {
            cudaGetLastError();
            return DEP_ERR_CUDA;
        }
        // The projection may start while the gather runs: it streams W first and
        // reads x only after waiting for the gather (the gather does not write W).
        // Kernels whose warps store runs of contiguous y bytes write it straight
        // into the mapped y_host (one kernel and one dependent-launch hop fewer
        // per call).  The cluster kernel stores y by bulk tensor copies from
        // shared memory into device memory, and the x-on-M kernel 32 bytes per
        // lane into 32 different rows, which over the host link took ~1.7x the
        // time of a copy (DSA at 32-256 rows, end to end: 473 against 274 us per
        // step): both write the staging area, and a copy kernel takes y back.
        // DEP_STAGING=stage takes that route for every kind (for comparisons).
        const bool direct = t && t->kind != DEP_KIND_TC_CLUSTER && t->kind != DEP_KIND_TC_XM &&
                            !env_is("DEP_STAGING", "stage");
        dep_status_t st = run_impl(plan, t, plan->x_stage, W, direct ? ay.devicePointer : plan->y_stage, B, stream,
                                   true);
        if (st != DEP_OK)
            return st;
        if (!direct && dep::stage_copy(plan->y_stage, static_cast<uint16_t *>(ay.devicePointer), (size_t)B * plan->N,
                                       true, s) != cudaSuccess) {
            cudaGetLastError();
            return DEP_ERR_CUDA;
        }
        return DEP_OK;
    }
    if (cudaMemcpyAsync(plan->x_stage, x_host, xb, cudaMemcpyHostToDevice, s) != cudaSuccess) {
        cudaGetLastError();
        return DEP_ERR_CUDA;
    }
    dep_status_t st = run_impl(plan, lookup(plan, B), plan->x_stage, W, plan->y_stage, B, stream);
    if (st != DEP_OK)
        return st;
    if (cudaMemcpyAsync(y_host, plan->y_stage, yb, cudaMemcpyDeviceToHost, s) != cudaSuccess) {
        cudaGetLastError();
        return DEP_ERR_CUDA;
    }
    return DEP_OK;
}

dep_status_t dep_projection_plan_query(dep_plan_t plan, int32_t B, dep_tactic_t *out)
{
    if (!plan || !out || B < 1)
        return DEP_ERR_INVALID_ARG;
    const dep_tactic_t *t = lookup(plan, B);
    if (!t)
        return DEP_ERR_INTERNAL;
    *out = *t;
    return DEP_OK;
}

dep_status_t dep_projection_plan_table(dep_plan_t plan, dep_tactic_t *out, int32_t cap, int32_t *n)
{
    if (!plan || !n || cap < 0 || (cap > 0 && !out))
        return DEP_ERR_INVALID_ARG;
    *n = (int32_t)plan->table.size();
    for (int32_t i = 0; i < cap && i < *n; ++i)
        out[i] = plan->table[(size_t)i];
    return DEP_OK;
}

dep_status_t dep_projection_plan_set(dep_plan_t plan, const dep_tactic_t *tactic)
{
    if (!plan || !tactic || !tactic_valid(*tactic))
        return DEP_ERR_INVALID_ARG;
    if (!plan->host_only && !grid_resident(*tactic, plan->N, plan->K, plan->sm_count))
        return DEP_ERR_UNSUPPORTED;
    const std::vector<dep_tactic_t> old = plan->table;
    bool replaced = false;
    for (auto &t : plan->table)
        if (t.max_rows == tactic->max_rows) {
            t = *tactic;
            replaced = true;
        }
    if (!replaced) {
        plan->table.push_back(*tactic);
        sort_table(plan->table);
    }
    if (!plan->host_only) {
        // Grow the workspace if the new entry needs more (synchronises the device).
        const dep_status_t st = allocate_device(plan);
        if (st != DEP_OK) {
            plan->table = old;
            return st;
        }
    }
    return DEP_OK;
}

dep_status_t dep_projection_plan_partials(dep_plan_t plan, void *host, size_t bytes, size_t *written)
{
    if (!plan || !written || (bytes && !host))
        return DEP_ERR_INVALID_ARG;
    *written = 0;
    if (plan->host_only)
        return DEP_ERR_UNSUPPORTED;
    const size_t n = std::min(bytes, plan->ws_floats * sizeof(float));
    if (cudaDeviceSynchronize() != cudaSuccess ||
        (n && cudaMemcpy(host, plan->ws, n, cudaMemcpyDeviceToHost) != cudaSuccess)) {
        cudaGetLastError();
        return DEP_ERR_CUDA;
    }
    *written = n;
    return DEP_OK;
}

dep_status_t dep_projection_plan_exchange(dep_plan_t plan, void *host, size_t bytes, size_t *written)
{
    if (!plan || !written || (bytes && !host))
        return DEP_ERR_INVALID_ARG;
    *written = 0;
    if (plan->host_only)
        return DEP_ERR_UNSUPPORTED;
    const size_t n = std::min(bytes, plan->xch_words * 8);
    if (cudaDeviceSynchronize() != cudaSuccess ||
        (n && cudaMemcpy(host, plan->xch, n, cudaMemcpyDeviceToHost) != cudaSuccess)) {
        cudaGetLastError();
        return DEP_ERR_CUDA;
    }
    *written = n;
    return DEP_OK;
}

dep_status_t dep_projection_plan_workspace(dep_plan_t plan, size_t *bytes)
{
    if (!plan || !bytes)
        return DEP_ERR_INVALID_ARG;
    *bytes = plan->dev_bytes;
    return DEP_OK;
}

dep_status_t dep_projection_plan_save(dep_plan_t plan, const char *path)
{
    if (!plan || !path)
        return DEP_ERR_INVALID_ARG;
    FILE *f = std::fopen(path, "w");
    if (!f)
        return DEP_ERR_IO;
    std::string name = plan->device_name;
    for (char &ch : name)
        if (ch == ' ' || ch == '\t' || ch == '\n')
            ch = '_';
    int ok = std::fprintf(f, "dep_projection_plan 2\ndevice %s\nsms %d\nshape %lld %lld\nentries %zu\n",
                          name.c_str(), plan->sm_count, (long long)plan->N, (long long)plan->K,
                          plan->table.size()) > 0;
    for (const auto &t : plan->table)
        ok = ok && std::fprintf(f, "%d %d %d %d %d %d %d %d\n", t.max_rows, t.kind, t.ctas, t.tile_n,
                                t.tile_k, t.stages, t.cols, t.splits) > 0;
    ok = (std::fclose(f) == 0) && ok;
    return ok ? DEP_OK : DEP_ERR_IO;
}

dep_status_t dep_projection_plan_load(const char *path, int64_t N, int64_t K, dep_plan_t *out)
{
    if (!out)
        return DEP_ERR_INVALID_ARG;
    *out = nullptr;
    if (!path)
        return DEP_ERR_INVALID_ARG;
    FILE *f = std::fopen(path, "r");
    if (!f)
        return DEP_ERR_IO;
    char name[512] = {0};
    int version = 0, sms = 0;
    long long fn = 0, fk = 0;
    size_t count = 0;
    std::vector<dep_tactic_t> table;
    bool ok = std::fscanf(f, "dep_projection_plan %d device %511s sms %d shape %lld %lld entries %zu",
                          &version, name, &sms, &fn, &fk, &count) == 6 &&
              (version == 1 || version == 2) && count >= 1 && count <= 4096;
    for (size_t i = 0; ok && i < count; ++i) {
        dep_tactic_t t{};  // version 1 files predate the K-piece field (0)
        ok = std::fscanf(f, "%d %d %d %d %d %d %d", &t.max_rows, &t.kind, &t.ctas, &t.tile_n,
                         &t.tile_k, &t.stages, &t.cols) == 7 &&
             (version == 1 || std::fscanf(f, "%d", &t.splits) == 1) && tactic_valid(t);
        table.push_back(t);
    }
    std::fclose(f);
    if (!ok)
        return DEP_ERR_IO;
    if (fn != N || fk != K)
        return DEP_ERR_INVALID_ARG;
    std::vector<int32_t> keys;
    for (const auto &t : table)
        keys.push_back(t.max_rows);
    dep_plan_t p = nullptr;
    dep_status_t st = make_plan(N, K, keys.data(), (int32_t)keys.size(), false, 0, &p);
    if (st != DEP_OK)
        return st;
    bool resident = true;
    for (const auto &t : table)
        resident = resident && grid_resident(t, N, K, p->sm_count);
    if (p->sm_count != sms || !resident) {
        dep_projection_plan_destroy(p);
        return DEP_ERR_UNSUPPORTED;
    }
    p->table = table;
    sort_table(p->table);
    st = allocate_device(p);
    if (st != DEP_OK) {
        dep_projection_plan_destroy(p);
        return st;
    }
    *out = p;
    return DEP_OK;
}

void dep_projection_plan_destroy(dep_plan_t plan)
{
    if (!plan)
        return;
    if (plan->dev_block) {
        int prev = -1;
        cudaGetDevice(&prev);
        cudaSetDevice(plan->device);
        cudaDeviceSynchronize();
        cudaFree(plan->dev_block);
        if (prev >= 0)
            cudaSetDevice(prev);
        cudaGetLastError();
    }
    delete plan;
}

dep_status_t dep_projection_device_status(dep_plan_t plan, void *stream, int32_t *code)
{
    if (!plan || !code)
        return DEP_ERR_INVALID_ARG;
    *code = 0;
    if (plan->host_only)
        return DEP_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int h = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemcpy(&h, plan->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(plan->status, 0, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return DEP_ERR_CUDA;
    }
    // After a give-up, counters and exchange flags may be left mid-protocol:
    // clear them so that the plan's next runs start from a clean state.
    if (h && (cudaDeviceSynchronize() != cudaSuccess ||
              cudaMemset(plan->counters, 0, plan->n_counters * sizeof(int) + plan->xch_words * 8) != cudaSuccess)) {
        cudaGetLastError();
        return DEP_ERR_CUDA;
    }
    *code = h;
    return h ? DEP_ERR_TIMEOUT : DEP_OK;
}

dep_status_t dep_projection_selftest_timeout(int32_t limit_us, int32_t *code)
{
    if (!code || limit_us < 1 || limit_us > 10000000)
        return DEP_ERR_INVALID_ARG;
    *code = 0;
    if (dep::selftest_timeout(limit_us, code) != cudaSuccess) {
        cudaGetLastError();
        return DEP_ERR_CUDA;
    }
    return DEP_OK;
}

dep_status_t dep_projection_plan_selftest_exchange(dep_plan_t plan, int32_t limit_us, void *stream)
{
    if (!plan || limit_us < 1 || limit_us > 10000000)
        return DEP_ERR_INVALID_ARG;
    if (plan->host_only)
        return DEP_ERR_UNSUPPORTED;
    if (plan->xch_words < 4 * 16 * 32 || plan->n_counters < 1)
        return DEP_ERR_UNSUPPORTED;  // a plan without tensor-core tactics has no exchange region
    if (dep::tcs_selftest_exchange(plan->xch, plan->xch_words, plan->counters, plan->status,
                                   (uint64_t)limit_us * 1000ull, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return DEP_ERR_CUDA;
    }
    return DEP_OK;
}

const char *dep_status_string(dep_status_t s)
{
    switch (s) {
    case DEP_OK: return "ok";
    case DEP_ERR_INVALID_ARG: return "invalid argument";
    case DEP_ERR_UNSUPPORTED: return "unsupported";
    case DEP_ERR_MISALIGNED: return "misaligned pointer or K not a multiple of 8";
    case DEP_ERR_CUDA: return "CUDA error";
    case DEP_ERR_OOM: return "out of device memory";
    case DEP_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
    case DEP_ERR_INTERNAL: return "internal error";
    case DEP_ERR_IO: return "plan file error";
    }
    return "unknown status";
}

int32_t dep_projection_version(void) { return 100; }

}  // extern "C"
