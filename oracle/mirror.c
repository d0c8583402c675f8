/*
 * mirror.c -- bit-exact FP32 replay of the split-K FMA tactic's summation order.
 *
 * TEST INFRASTRUCTURE ONLY (same rules as oracle.c: the product never loads it,
 * and it shares no code with the CUDA path).
 *
 * The pages fix the arithmetic types (runtime.dep page, module overview,
 * precision paragraph: FP32 accumulation, BF16 outputs) and say the split-K
 * order differs from the stock GEMM's without giving it (runtime.hybrid page,
 * HybridAttention.__init__: warp split-K up to 16 rows).  The library fixes one
 * order per tactic so that results are reproducible bit for bit; this file
 * restates that order for the FMA tactic in plain C, so that a GPU result can be
 * compared with it for equality rather than within a tolerance.
 *
 * The order, for a grid of C persistent blocks, blocks of RB weight rows and
 * k-tiles of KT = 32 * 8 columns:
 *   units      u = t * KTILES + kt,  t < ceil(N/RB) row blocks, kt < ceil(K/KT)
 *   block c    owns units [floor(c U / C), floor((c+1) U / C)),  U = #units
 *   segment    the units one block owns inside one row block (consecutive kt)
 *   lane l     of a warp owns columns kt*KT + 8 l + j, j = 0..7, of every tile
 *   lane chain acc = +0; for each kt of the segment, for j = 0..7:
 *                acc = fmaf(w, x, acc)   (w, x = +0 past column K-1)
 *   warp sum   butterfly over lanes with offsets 16, 8, 4, 2, 1: v += v[lane^off]
 *   split sum  the segments of a row block, in increasing block order:
 *                s = p0; s = s + p1; ...   (one segment: s = p0)
 *   output     round s to BF16, nearest, ties to even.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static float mir_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16; /* BF16 is the top half of an FP32 */
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint16_t mir_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))
        return (uint16_t)(0x7FC0); /* any NaN: canonical quiet NaN */
    /* nearest, ties to even: add half an ulp minus one, plus the kept lsb */
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* Block that owns unit u in the balanced split of U units over C blocks. */
static int64_t mir_owner(int64_t u, int64_t U, int64_t C)
{
    int64_t c = (u * C) / U; /* first guess, then step to the exact owner */
    while (c > 0 && (c * U) / C > u)
        --c;
    while (c + 1 < C && ((c + 1) * U) / C <= u)
        ++c;
    return c;
}

/* Partial of one segment: rows' k-tiles [kt0, kt1) for output (b, n). */
static float mir_segment(const uint16_t *xr, const uint16_t *wr, int64_t K,
                         int64_t kt0, int64_t kt1, int KT)
{
    float v[32];
    int per_lane = KT / 32;
    for (int l = 0; l < 32; ++l) {
        float acc = 0.0f;
        for (int64_t kt = kt0; kt < kt1; ++kt)
            for (int j = 0; j < per_lane; ++j) {
                int64_t k = kt * KT + (int64_t)l * per_lane + j;
                float w = k < K ? mir_f32(wr[k]) : 0.0f;
                float a = k < K ? mir_f32(xr[k]) : 0.0f;
                acc = fmaf(w, a, acc);
            }
        v[l] = acc;
    }
    for (int off = 16; off >= 1; off >>= 1) {
        float t[32];
        for (int l = 0; l < 32; ++l)
            t[l] = v[l] + v[l ^ off];
        memcpy(v, t, sizeof v);
    }
    return v[0];
}

/* y[B,N] by the FMA tactic's order for a grid of `ctas` blocks of `rows` weight
 * rows and k-tiles of `KT` columns.  Returns 0, or -1 on bad arguments. */
int mirror_fma_linear(const uint16_t *x, const uint16_t *W, uint16_t *y,
                      int64_t B, int64_t N, int64_t K, int ctas, int rows, int KT,
                      int threads)
{
    if (B < 0 || N < 0 || K < 0 || ctas < 1 || rows < 1 || KT < 32 || KT % 32)
        return -1;
    if (B == 0 || N == 0)
        return 0;
    int64_t T = (N + rows - 1) / rows, KTILES = (K + KT - 1) / KT;
    if (KTILES == 0)
        KTILES = 1; /* K = 0: one all-padding tile, the sums are +0 */
    int64_t U = T * KTILES, C = ctas;
#ifdef _OPENMP
    if (threads <= 0)
        threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 8) num_threads(threads)
#endif
    for (int64_t i = 0; i < B * N; ++i) {
        int64_t b = i / N, n = i % N, t = n / rows;
        int64_t first = t * KTILES, last = first + KTILES - 1;
        int64_t c0 = mir_owner(first, U, C), c1 = mir_owner(last, U, C);
        float s = 0.0f;
        for (int64_t c = c0; c <= c1; ++c) {
            int64_t u0 = (c * U) / C, u1 = ((c + 1) * U) / C;
            if (u0 < first)
                u0 = first;
            if (u1 > last + 1)
                u1 = last + 1;
            if (u0 >= u1)
                continue; /* a block with no unit in this row block */
            float p = mir_segment(x + b * K, W + n * K, K, u0 - first, u1 - first, KT);
            s = (c == c0) ? p : s + p;
        }
        y[i] = mir_bf16(s);
    }
    (void)threads;
    return 0;
}
