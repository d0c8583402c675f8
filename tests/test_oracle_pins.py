"""Pins of the CPU oracle against facts fixed by the pages and by arithmetic.

The oracle computes y = RNE_bf16(exact sum_k x[b,k] W[n,k]) (runtime.dep page,
DepProjection; precision paragraph of its module overview).  Each test below
checks it against something other than itself: hand-derived worked examples,
exact rational arithmetic on tiny shapes, closed forms, invariants of the exact
sum, an exhaustive sweep of BF16 bit patterns, and a float64 matmul.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

from helpers import bf16_fraction, exact_bf16, rne_bf16_fraction, within_tolerance
from skinny_bf16_split_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.txt")


def _examples():
    blocks, cur = [], {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, rest = line.partition(" ")
        if key == "name":
            if cur:
                blocks.append(cur)
            cur = {"name": rest}
        else:
            cur[key] = rest.split()
    blocks.append(cur)
    return blocks


@pytest.mark.parametrize("ex", _examples(), ids=lambda e: e["name"])
def test_worked_examples(orc, ex):
    B, N, K = (int(v) for v in ex["shape"])
    x = np.array([exact_bf16(float(v)) for v in ex["x"]], dtype=np.uint16).reshape(B, K)
    W = np.array([exact_bf16(float(v)) for v in ex["W"]], dtype=np.uint16).reshape(N, K)
    want = np.array([int(v, 16) for v in ex["y"]], dtype=np.uint16).reshape(B, N)
    np.testing.assert_array_equal(orc.linear(x, W), want)


def test_identity_exhaustive(orc):
    """x * 1.0 over every BF16 bit pattern returns it (0 -> +0, NaN -> 0x7FC0)."""
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(-1, 1)
    y = orc.linear(h, np.array([[0x3F80]], dtype=np.uint16))[:, 0]
    f = synth.bf16_to_f32(h[:, 0])
    want = h[:, 0].copy()
    want[np.isnan(f)] = 0x7FC0
    want[f == 0] = 0x0000
    np.testing.assert_array_equal(y, want)


@pytest.mark.parametrize("factor_bits,factor", [(0x4000, 2), (0x3F00, Fraction(1, 2)),
                                                (0x3E80, Fraction(1, 4)),
                                                (0xBFC0, Fraction(-3, 2))])
def test_scaling_exhaustive(orc, factor_bits, factor):
    """Every finite BF16 times a constant: matches exact rational RNE, including
    the subnormal range (halving drops bits there) and overflow to infinity."""
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = synth.bf16_to_f32(h)
    h = h[np.isfinite(f)]
    y = orc.linear(h.reshape(-1, 1), np.array([[factor_bits]], dtype=np.uint16))[:, 0]
    rng = np.random.default_rng(1)
    sel = np.concatenate([np.arange(0, 300), np.arange(len(h) - 300, len(h)),
                          rng.choice(len(h), 3000, replace=False)])
    for i in sel:
        want = rne_bf16_fraction(bf16_fraction(h[i]) * factor)
        assert int(y[i]) == want, (hex(h[i]), hex(y[i]), hex(want))


def test_fraction_bruteforce(orc):
    """Tiny random shapes with values across the whole BF16 exponent range,
    against exact rational sums rounded by an independent RNE."""
    rng = np.random.default_rng(2024)
    for trial in range(60):
        B, N, K = rng.integers(1, 5), rng.integers(1, 9), rng.integers(1, 17)
        # random finite patterns, exponent fields limited so sums cannot overflow
        def draw(shape):
            sign = rng.integers(0, 2, shape) << 15
            field = rng.integers(0, 190, shape)  # includes subnormals (field 0)
            if trial % 3 == 0:
                field = rng.integers(100, 140, shape)  # similar magnitudes: cancellation
            frac = rng.integers(0, 128, shape)
            return (sign | (field << 7) | frac).astype(np.uint16)
        x, W = draw((B, K)), draw((N, K))
        y = orc.linear(x, W)
        for b in range(B):
            for n in range(N):
                s = sum(bf16_fraction(x[b, k]) * bf16_fraction(W[n, k]) for k in range(K))
                assert int(y[b, n]) == rne_bf16_fraction(s), (trial, b, n)


def test_closed_form_all_ones(orc):
    """All-ones x gives BF16(row sums of W), row sums taken exactly."""
    W = synth.normal_bf16(11, 1, (24, 300), sigma=0.02)
    x = np.full((3, 300), 0x3F80, dtype=np.uint16)
    y = orc.linear(x, W)
    for n in range(24):
        want = rne_bf16_fraction(sum(bf16_fraction(v) for v in W[n]))
        assert (y[:, n] == want).all()


def test_closed_form_identity_and_one_hot(orc):
    """W = [I_N | 0] returns x[:, :N]; one-hot rows select columns of x."""
    N, K = 40, 64
    x = synth.normal_bf16(3, 2, (5, K))
    W = np.zeros((N, K), dtype=np.uint16)
    W[np.arange(N), np.arange(N)] = 0x3F80
    xz = x[:, :N].copy()
    xz[synth.bf16_to_f32(xz) == 0] = 0  # -0 * 1 sums to +0
    np.testing.assert_array_equal(orc.linear(x, W), xz)
    cols = np.random.default_rng(5).integers(0, K, N)
    W = np.zeros((N, K), dtype=np.uint16)
    W[np.arange(N), cols] = 0x3F80
    np.testing.assert_array_equal(orc.linear(x, W), x[:, cols])


def test_invariants(orc):
    """Negation, power-of-two scaling, joint K permutation and N permutation."""
    B, N, K = 4, 50, 777
    x = synth.normal_bf16(9, 2, (B, K))
    W = synth.normal_bf16(9, 1, (N, K), sigma=0.02)
    y = orc.linear(x, W)
    nz = synth.bf16_to_f32(y) != 0
    # y(-x) = -y(x): flip sign bits of x; nonzero outputs flip sign bits exactly
    yn = orc.linear(x ^ np.uint16(0x8000), W)
    np.testing.assert_array_equal(yn[nz], y[nz] ^ np.uint16(0x8000))
    # y(2^3 x) = 2^3 y(x): add 3 to every nonzero exponent field (no overflow here)
    f = synth.bf16_to_f32(x)
    assert np.abs(f).max() < 2.0 ** 100 and np.abs(f[f != 0]).min() > 2.0 ** -100
    x8 = np.where(f != 0, x + np.uint16(3 << 7), x).astype(np.uint16)
    y8 = orc.linear(x8, W)
    fy = synth.bf16_to_f32(y)
    assert np.abs(fy[fy != 0]).min() > 2.0 ** -100
    np.testing.assert_array_equal(y8[nz], (y[nz] + np.uint16(3 << 7)).astype(np.uint16))
    # joint K permutation: the exact sum does not depend on the order
    perm = np.random.default_rng(0).permutation(K)
    np.testing.assert_array_equal(orc.linear(x[:, perm], W[:, perm]), y)
    # N permutation permutes the outputs
    pn = np.random.default_rng(1).permutation(N)
    np.testing.assert_array_equal(orc.linear(x, W[pn]), y[:, pn])


def test_linearity(orc):
    """y(x1 + x2) = y(x1) + y(x2) up to the three output roundings."""
    K = 512
    x1 = synth.normal_bf16(1, 2, (2, K))
    x2 = synth.normal_bf16(2, 2, (2, K))
    W = synth.normal_bf16(3, 1, (64, K), sigma=0.02)
    xs = synth.bf16_from_f64(synth.bf16_to_f32(x1).astype(np.float64)
                             + synth.bf16_to_f32(x2).astype(np.float64))
    # only where x1 + x2 was exact in BF16 is linearity of the exact sum testable
    exact = (synth.bf16_to_f32(xs).astype(np.float64)
             == synth.bf16_to_f32(x1).astype(np.float64) + synth.bf16_to_f32(x2).astype(np.float64))
    x1 = np.where(exact, x1, 0).astype(np.uint16)
    x2 = np.where(exact, x2, 0).astype(np.uint16)
    xs = np.where(exact, xs, 0).astype(np.uint16)
    ys = synth.bf16_to_f32(orc.linear(xs, W)).astype(np.float64)
    y1 = synth.bf16_to_f32(orc.linear(x1, W)).astype(np.float64)
    y2 = synth.bf16_to_f32(orc.linear(x2, W)).astype(np.float64)
    # each of the three roundings is off by at most half an ulp = 2^-8 relative
    # to its own value, and the exact sums are linear
    assert np.all(np.abs(ys - (y1 + y2)) <= 2.0 ** -8 * (np.abs(ys) + np.abs(y1) + np.abs(y2)))


def test_matches_float64_matmul(orc):
    """On N(0, .) inputs the exact oracle equals a float64 matmul rounded once to
    BF16 by an independent rounding routine (double error is far below half a
    BF16 ulp at these sizes)."""
    for seed, (B, N, K) in enumerate([(3, 257, 1000), (16, 130, 7168), (1, 2000, 12288)]):
        x = synth.normal_bf16(seed, 2, (B, K))
        W = synth.normal_bf16(seed, 1, (N, K), sigma=0.02)
        ref = synth.bf16_from_f64(synth.bf16_to_f32(x).astype(np.float64)
                                  @ synth.bf16_to_f32(W).astype(np.float64).T)
        np.testing.assert_array_equal(orc.linear(x, W), ref)


def test_special_values(orc):
    one, inf, ninf, nan, zero = 0x3F80, 0x7F80, 0xFF80, 0x7FC1, 0x0000
    big = 0x7F7F  # largest finite BF16
    cases = [
        ([nan, one], [one, one], 0x7FC0),      # NaN propagates (canonical)
        ([inf, one], [zero, one], 0x7FC0),     # Inf * 0
        ([inf, ninf], [one, one], 0x7FC0),     # +Inf + -Inf
        ([inf, one], [one, one], 0x7F80),      # Inf dominates
        ([ninf, one], [one, one], 0xFF80),
        ([big, big], [one, one], 0x7F80),      # overflow after summation
        ([big, big ^ 0x8000], [one, one], 0x0000),  # exact cancellation -> +0
    ]
    for xv, wv, want in cases:
        y = orc.linear(np.array([xv], dtype=np.uint16), np.array([wv], dtype=np.uint16))
        assert int(y[0, 0]) == want, (xv, wv, hex(y[0, 0]))


def test_statistics_of_workload_shapes(orc):
    """N(0,1) x and N(0,0.02) W: y has standard deviation about 0.02 sqrt(K)."""
    for K in (7168, 12288):
        x = synth.normal_bf16(0, 2, (2, K))
        W = synth.normal_bf16(0, 1, (512, K), sigma=0.02)
        sd = synth.bf16_to_f32(orc.linear(x, W)).std()
        assert abs(sd / (0.02 * np.sqrt(K)) - 1) < 0.1


def test_rows_subset_matches_full(orc):
    x = synth.normal_bf16(4, 2, (3, 640))
    W = synth.normal_bf16(4, 1, (300, 640), sigma=0.02)
    rows = np.array([0, 7, 299, 150, 7])
    np.testing.assert_array_equal(orc.linear_rows(x, W, rows), orc.linear(x, W)[:, rows])


def test_rms_rows_generator():
    x = synth.rms_rows_bf16(0, 2, (3, 7168))
    f = synth.bf16_to_f32(x).astype(np.float64)
    assert np.allclose(np.sqrt((f * f).mean(axis=1)), 1.0, atol=2e-3)


def test_generator_rounding_matches_rational_rne():
    """The input generator's float64 -> BF16 rounding against exact rationals."""
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-45, 38, 2000),
                        [0.0, -0.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 2.0 ** -133, 2.0 ** -134,
                         3 * 2.0 ** -135, 3.3961e38, -3.3961e38, 1e39]])
    got = synth.bf16_from_f64(v)
    for vi, gi in zip(v, got):
        want = rne_bf16_fraction(Fraction(float(vi))) if vi != 0 else (0x8000 if np.signbit(vi) else 0)
        assert int(gi) == want, (vi, hex(gi), hex(want))


def test_tolerance_helper_rejects_a_wrong_answer(orc):
    """The acceptance bound is tight enough to see a one-term error."""
    x = synth.normal_bf16(5, 2, (2, 1024))
    W = synth.normal_bf16(5, 1, (64, 1024), sigma=0.02)
    y = orc.linear(x, W)
    assert within_tolerance(y, y)[0]
    bad = orc.linear(x[:, 1:], W[:, 1:])  # one dropped term
    Wt = W.copy()
    Wt[:, 3] ^= np.uint16(0x8000)        # one wrong sign
    assert not within_tolerance(bad, y)[0] or not within_tolerance(orc.linear(x, Wt), y)[0]


# --- the FP32 mirror of the FMA tactic ---------------------------------------

@pytest.mark.parametrize("ctas,rows", [(1, 64), (7, 64), (152, 64), (152, 32), (1000, 8)])
def test_mirror_within_tolerance_of_oracle(orc, ctas, rows):
    B, N, K = 4, 333, 3000
    x = synth.normal_bf16(6, 2, (B, K))
    W = synth.normal_bf16(6, 1, (N, K), sigma=0.02)
    ok, worst, idx = within_tolerance(orc.mirror_fma(x, W, ctas, rows), orc.linear(x, W))
    assert ok, (worst, idx)


def test_mirror_exact_on_small_integers(orc):
    """Small-integer inputs: every partial sum is an exact integer in FP32, so
    any summation order gives the exact result."""
    rng = np.random.default_rng(3)
    B, N, K = 3, 70, 600
    xi = rng.integers(-16, 17, (B, K))
    wi = rng.integers(-16, 17, (N, K))
    x = np.array([exact_bf16(v) for v in xi.ravel()], dtype=np.uint16).reshape(B, K)
    W = np.array([exact_bf16(v) for v in wi.ravel()], dtype=np.uint16).reshape(N, K)
    want = synth.bf16_from_f64((xi @ wi.T).astype(np.float64))
    np.testing.assert_array_equal(orc.linear(x, W), want)
    for ctas in (1, 5, 152):
        np.testing.assert_array_equal(orc.mirror_fma(x, W, ctas, 32), want)


def test_mirror_order_is_not_the_exact_sum(orc):
    """The mirror really sums in FP32: a cancellation the exact oracle resolves
    is lost when the large terms meet first in one lane's chain."""
    K = 256
    xv = np.zeros(K)
    xv[0], xv[1], xv[2] = 2.0 ** 30, 1.0, -(2.0 ** 30)  # lane 0 holds k = 0..7
    x = np.array([[exact_bf16(v) for v in xv]], dtype=np.uint16)
    W = np.full((1, K), 0x3F80, dtype=np.uint16)
    assert int(orc.linear(x, W)[0, 0]) == 0x3F80
    assert int(orc.mirror_fma(x, W, 1, 8)[0, 0]) == 0x0000
