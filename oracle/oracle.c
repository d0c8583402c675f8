/*
 * oracle.c -- exact CPU oracle for the decode projection  y = BF16( x . W^T ).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may load, call or link
 * this file; only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (the plain definition of the method's result):
 *   runtime.dep page, DepProjection: a TP1 linear whose output is the product of
 *   the activation rows x[B,K] with the transposed weight W[N,K], written into a
 *   caller-owned BF16 buffer y[B,N] (the cuBLAS branch is torch.mm(x, W.t())).
 *   runtime.dep page, module overview (precision paragraph) and runtime.hybrid
 *   page, module overview: BF16 inputs, FP32 accumulation, BF16 outputs; the
 *   split-K summation order differs from the stock GEMM.
 * Since the order of the FP32 sum is left open, the one order-free result is the
 * exact real sum, rounded once to BF16.  That is what this oracle returns:
 *
 *   y[b,n] = RNE_bf16( sum_k x[b,k] * W[n,k] )   (exact sum, one rounding)
 *
 * How it is exact.  A finite BF16 value is M * 2^E with an integer significand
 * M in [0,255] and E in [-133,120] (normal: M = 128 + fraction, E = field - 134;
 * subnormal: M = fraction, E = -133).  A product of two of them is the integer
 * M1*M2 < 2^16 times 2^(E1+E2) with E1+E2 >= -266, so every product is an
 * integer multiple of 2^-266.  The sum is accumulated as a signed fixed-point
 * integer with LSB 2^-266 in 32-bit limbs held in int64 (carries deferred), which
 * loses nothing for any K below 2^31.  The exact sum is then rounded once to BF16,
 * round to nearest, ties to even (the IEEE 754 default rounding attribute).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - rounding mode of the BF16 output: round to nearest, ties to even;
 *   - an exact zero sum is returned as +0;
 *   - non-finite inputs follow IEEE semantics: NaN in, Inf*0, or +Inf with -Inf
 *     gives the canonical quiet NaN 0x7FC0; otherwise any Inf term gives that Inf;
 *   - overflow past the largest finite BF16 (after rounding) gives +-Inf.
 */
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_LIMBS 20        /* 640 bits: products reach bit 506, sums < 2^(506+16+31) */
#define ORC_LSB_EXP (-266)  /* weight of bit 0 of the accumulator */

/* Decode BF16 bits into (class, sign, M, E) with value = (-1)^sign * M * 2^E.
 * class: 0 finite, 1 infinity, 2 NaN.  Follows the binary16-brain layout:
 * 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
typedef struct { int cls, sign, M, E; } orc_bf16_t;

static orc_bf16_t orc_decode(uint16_t h)
{
    orc_bf16_t d;
    int field = (h >> 7) & 0xFF, frac = h & 0x7F;
    d.sign = h >> 15;
    if (field == 0xFF) {
        d.cls = frac ? 2 : 1;
        d.M = 0;
        d.E = 0;
    } else if (field == 0) {
        d.cls = 0;
        d.M = frac;
        d.E = -133;
    } else {
        d.cls = 0;
        d.M = 128 + frac;
        d.E = field - 134;
    }
    return d;
}

/* Round the exact value (-1)^neg * A * 2^-266 (A = non-negative multi-limb
 * integer, 32 bits per limb, little-endian) to BF16, ties to even. */
static uint16_t orc_round(int neg, const uint32_t *A)
{
    int p = -1; /* index of the highest set bit */
    for (int i = ORC_LIMBS - 1; i >= 0 && p < 0; --i)
        if (A[i])
            for (int b = 31; b >= 0; --b)
                if ((A[i] >> b) & 1u) { p = 32 * i + b; break; }
    if (p < 0)
        return 0x0000; /* exact zero: +0 */

    /* Bit index of the result's unit in the last place: 8 significant bits for a
     * normal result, the fixed subnormal quantum 2^-133 (bit 133) otherwise. */
    int q = p - 7;
    if (q < 133)
        q = 133;

    uint32_t M = 0; /* bits [q, q+7] of A: the 8 kept significand bits */
    for (int j = 7; j >= 0; --j) {
        int bit = q + j;
        M = (M << 1) | ((A[bit / 32] >> (bit % 32)) & 1u);
    }
    int round_bit = (A[(q - 1) / 32] >> ((q - 1) % 32)) & 1u;
    int sticky = 0;
    for (int bit = 0; bit < q - 1 && !sticky; ++bit)
        sticky = (A[bit / 32] >> (bit % 32)) & 1u;

    if (round_bit && (sticky || (M & 1u)))
        M += 1;
    if (M == 256) { /* carried into a new binade */
        M = 128;
        q += 1;
    }
    uint16_t s = (uint16_t)(neg ? 0x8000 : 0);
    if (q == 133 && M < 128)
        return (uint16_t)(s | M); /* subnormal (or zero after rounding: impossible here) */
    int field = q - 132;          /* value = M * 2^(q-266) = (M/128) * 2^(field-127) */
    if (field >= 255)
        return (uint16_t)(s | 0x7F80); /* overflow: infinity */
    return (uint16_t)(s | (field << 7) | (M - 128));
}

/* One output element: exact dot product of x row b and W row n, rounded once. */
static uint16_t orc_dot(const uint16_t *xr, const uint16_t *wr, int64_t K)
{
    int64_t acc[ORC_LIMBS];
    memset(acc, 0, sizeof acc);
    int nan = 0, pinf = 0, ninf = 0;
    for (int64_t k = 0; k < K; ++k) {
        orc_bf16_t a = orc_decode(xr[k]), w = orc_decode(wr[k]);
        int sign = a.sign ^ w.sign;
        if (a.cls == 2 || w.cls == 2) { nan = 1; continue; }
        if (a.cls == 1 || w.cls == 1) {
            /* Inf times zero is NaN; Inf times nonzero is a signed infinity. */
            if ((a.cls == 0 && a.M == 0) || (w.cls == 0 && w.M == 0))
                nan = 1;
            else if (sign)
                ninf = 1;
            else
                pinf = 1;
            continue;
        }
        uint64_t m = (uint64_t)a.M * (uint64_t)w.M; /* < 2^16, exact */
        if (!m)
            continue;
        int off = a.E + w.E - ORC_LSB_EXP; /* 0 .. 506 */
        uint64_t v = m << (off % 32);     /* < 2^48: spans two limbs */
        int limb = off / 32;
        int64_t lo = (int64_t)(v & 0xFFFFFFFFu), hi = (int64_t)(v >> 32);
        if (sign) { lo = -lo; hi = -hi; }
        acc[limb] += lo;
        acc[limb + 1] += hi;
    }
    if (nan || (pinf && ninf))
        return 0x7FC0;
    if (pinf)
        return 0x7F80;
    if (ninf)
        return 0xFF80;

    /* Propagate carries so that every limb but the top one is in [0, 2^32). */
    for (int i = 0; i < ORC_LIMBS - 1; ++i) {
        int64_t c = acc[i] >> 32; /* arithmetic shift = floor division by 2^32 */
        acc[i] -= c * ((int64_t)1 << 32);
        acc[i + 1] += c;
    }
    /* Two's-complement value sum acc[i] 2^(32 i); take sign and magnitude. */
    int neg = acc[ORC_LIMBS - 1] < 0;
    uint32_t A[ORC_LIMBS];
    if (!neg) {
        for (int i = 0; i < ORC_LIMBS; ++i)
            A[i] = (uint32_t)acc[i];
    } else {
        /* magnitude = -value: complement every limb and add one */
        uint64_t carry = 1;
        for (int i = 0; i < ORC_LIMBS; ++i) {
            uint64_t limb = (uint64_t)(~(uint32_t)acc[i]) + carry;
            A[i] = (uint32_t)limb;
            carry = limb >> 32;
        }
    }
    return orc_round(neg, A);
}

/* y[b*N + n] = RNE_bf16(sum_k x[b*K+k] W[n*K+k]) for all b < B, n < N.
 * x, W, y are BF16 bit patterns, row-major and contiguous. threads <= 0: all. */
void oracle_linear(const uint16_t *x, const uint16_t *W, uint16_t *y,
                   int64_t B, int64_t N, int64_t K, int threads)
{
#ifdef _OPENMP
    if (threads <= 0)
        threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 16) num_threads(threads)
#endif
    for (int64_t i = 0; i < B * N; ++i) {
        int64_t b = i / N, n = i % N;
        y[i] = orc_dot(x + b * K, W + n * K, K);
    }
    (void)threads;
}

/* The same for a subset of weight rows: y_rows[b*R + r] is output (b, rows[r]).
 * Used to check sampled outputs of full-size problems. */
void oracle_linear_rows(const uint16_t *x, const uint16_t *W, const int64_t *rows,
                        int64_t R, uint16_t *y_rows, int64_t B, int64_t K, int threads)
{
#ifdef _OPENMP
    if (threads <= 0)
        threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 4) num_threads(threads)
#endif
    for (int64_t i = 0; i < B * R; ++i) {
        int64_t b = i / R, r = i % R;
        y_rows[i] = orc_dot(x + b * K, W + rows[r] * K, K);
    }
    (void)threads;
}

/* Threads an OpenMP region of this library would use by default. */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
