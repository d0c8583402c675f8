"""The x-on-M tensor-core tactic (DEP_KIND_TC_XM) against the oracle.

Batch rows are the MMA's M side (blocks of 128 rows, or 64 for a pass of at
most 64 rows), tiles of R weight rows its N side; every block sums its tiles'
whole K, or a pair of blocks (a cluster of two) shares a tile, each half of K,
the halves added in order through distributed shared memory; two issuers each
into its own accumulator.  Checked here: the
acceptance tolerance against the exact oracle for tiles of 16 to 256 rows, one
to four slices per stage, one or two blocks of rows per pass (passes of <= 64,
<= 128, <= 256 rows and several passes), ragged N, K and B, grids of 1, 7 and
all SMs; identical bits whatever the grid, the ring depth and the stage width
(the same MMA chains in the same order); exact small-integer sums; sign
symmetry; run-to-run and CUDA-graph determinism on the full DSA shape; the
same for pairs, whose bits depend on neither the number of pairs, the depth nor
the stage width.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gpu_util import empty_out, to_dev, to_host  # noqa: E402
from helpers import exact_bf16, within_tolerance  # noqa: E402
from skinny_bf16_split_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu

SMEM_MAX = 227 * 1024


def sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


def deepest(R, tile_k, cols, want=16, pair=False):
    """Deepest ring (at most `want`) of the tactic at 128-row x blocks (pairs: one
    whose ring at 64-row x blocks also holds the other CTA's partials)."""
    atoms, mb = tile_k // 64, cols // 128
    best = 0
    for st in range(2, want + 1):
        if 1024 + st * atoms * (R + mb * 128) * 128 + (2 * st + 8) * 8 + 16 > SMEM_MAX:
            continue
        if pair and mb * 128 * (R // 2) * 4 > st * atoms * (R + mb * 64) * 128:
            continue
        best = st
    return best


def xm_tactic(dep, R, cols, tile_k, stages, ctas, max_rows=None, pair=False):
    return dep.dep_tactic_t(max_rows=max_rows or cols, kind=dep.DEP_KIND_TC_XM, ctas=ctas, tile_n=R,
                            tile_k=tile_k, stages=stages, cols=cols, splits=2 if pair else 0)


def run(dep, plan, x, W, N, tactic):
    B = x.shape[0]
    y = empty_out(B, N)
    dep.dep_projection_run_tactic(plan, tactic, to_dev(x), to_dev(W), y, B)
    torch.cuda.synchronize()
    return to_host(y)


@pytest.fixture(scope="module")
def plans(dep):
    cache = {}

    def get(N, K):
        if (N, K) not in cache:
            cache[(N, K)] = dep.dep_projection_plan(N, K, [256])
        return cache[(N, K)]

    yield get
    for p in cache.values():
        assert dep.dep_projection_device_status(p) == 0
        dep.dep_projection_plan_destroy(p)


_refs = {}


def inputs_and_ref(orc, N, K, B):
    """Seeded inputs of one shape and the oracle's result (computed once)."""
    if (N, K, B) not in _refs:
        W = synth.normal_bf16(N + K, 1, (N, K), sigma=0.02)
        x = synth.normal_bf16(N + B, 2, (B, K))
        _refs[(N, K, B)] = (x, W, orc.linear(x, W))
    return _refs[(N, K, B)]


@pytest.mark.parametrize("N,K", [(333, 1000), (97, 264), (1000, 3136), (700, 2048)])
@pytest.mark.parametrize("R", [16, 48, 96, 112, 256])
def test_xm_parity_vs_oracle(dep, orc, plans, N, K, R):
    """Tiles of R weight rows (the last one ragged); passes of <= 64 rows (MMA
    M = 64), <= 128 and <= 256 rows and several passes; one or two blocks of 128
    rows per pass; 1, 2 or 4 slices per stage (K = 1000 and 264: one copy per
    slice, a ragged last slice; K = 3136: one copy per stage, the last stage
    partly past K; K = 2048: whole stages); grids of 1, 7 and all SMs."""
    plan = plans(N, K)
    for B in (17, 64, 100, 129, 300):
        x, W, ref = inputs_and_ref(orc, N, K, B)
        for cols in (128, 256):
            for tile_k in (64, 128, 256):
                st = deepest(R, tile_k, cols)
                if not st:
                    continue
                for ctas in (1, 7, sm_count()):
                    y = run(dep, plan, x, W, N, xm_tactic(dep, R, cols, tile_k, st, ctas))
                    ok, worst, idx = within_tolerance(y, ref)
                    assert ok, (B, cols, tile_k, st, ctas, worst, idx)


@pytest.mark.parametrize("cols,B", [(128, 40), (128, 128), (256, 200), (128, 300), (256, 64)])
def test_xm_bits_independent_of_grid_depth_and_stage_width(dep, plans, cols, B):
    """Every output is the same MMA chains in the same K order whatever the grid
    (tiles dealt to blocks), the ring depth and the slices per stage: identical
    bits."""
    N, K, R = 1000, 3072, 96
    plan = plans(N, K)
    W = synth.normal_bf16(31, 1, (N, K), sigma=0.02)
    x = synth.normal_bf16(32, 2, (B, K))
    ref = run(dep, plan, x, W, N, xm_tactic(dep, R, cols, 128, deepest(R, 128, cols), sm_count()))
    for tile_k in (64, 128, 256):
        top = deepest(R, tile_k, cols)
        for st in sorted({2, top}) if top else ():  # the shallowest and deepest rings that fit
            for ctas in (1, 5, sm_count()):
                y = run(dep, plan, x, W, N, xm_tactic(dep, R, cols, tile_k, st, ctas))
                np.testing.assert_array_equal(y, ref, err_msg=str((tile_k, st, ctas)))


def test_xm_small_integers_exact(dep, orc, plans):
    """Small-integer inputs give exact FP32 sums: every tactic equals the exact
    oracle bit for bit."""
    rng = np.random.default_rng(29)
    N, K = 700, 2048
    x = np.vectorize(exact_bf16)(rng.integers(-8, 9, (300, K))).astype(np.uint16)
    W = np.vectorize(exact_bf16)(rng.integers(-8, 9, (N, K))).astype(np.uint16)
    plan = plans(N, K)
    for B in (33, 128, 300):
        ref = orc.linear(x[:B], W)
        for R, cols, tile_k in ((96, 128, 128), (48, 256, 64), (256, 128, 64)):
            y = run(dep, plan, x[:B], W, N, xm_tactic(dep, R, cols, tile_k, deepest(R, tile_k, cols), 7))
            np.testing.assert_array_equal(y, ref, err_msg=str((B, R, cols, tile_k)))


def test_xm_negation_symmetric(dep, plans):
    """y(-x) = -y(x) bit for bit: every FP32 step, the two issuers' sum included,
    is sign-symmetric."""
    N, K = 900, 4096
    plan = plans(N, K)
    W = synth.normal_bf16(37, 1, (N, K), sigma=0.02)
    for B, cols in ((60, 128), (128, 128), (256, 256)):
        x = synth.normal_bf16(37 + B, 2, (B, K))
        t = xm_tactic(dep, 96, cols, 128, deepest(96, 128, cols), sm_count())
        y = run(dep, plan, x, W, N, t)
        yn = run(dep, plan, x ^ np.uint16(0x8000), W, N, t)
        nz = synth.bf16_to_f32(y) != 0
        np.testing.assert_array_equal(yn[nz], y[nz] ^ np.uint16(0x8000))


@pytest.mark.parametrize("B", [32, 64, 128])
def test_xm_default_plan_determinism_and_graph_replay(dep, orc, B):
    """The default plan of the DSA input projection (14560 x 7168) takes this
    kind from 32 to 128 rows; repeated runs and CUDA-graph replays give
    identical bits, within tolerance of the oracle on sampled rows."""
    N, K = 14560, 7168
    plan = dep.dep_projection_plan(N, K, [B])
    try:
        assert dep.dep_projection_plan_query(plan, B).kind == dep.DEP_KIND_TC_XM
        W = synth.normal_bf16(41, 1, (N, K), sigma=0.02)
        x = synth.normal_bf16(42, 2, (B, K))
        xd, Wd = to_dev(x), to_dev(W)
        ys = [empty_out(B, N) for _ in range(3)]
        for y in ys:
            dep.dep_projection_run(plan, xd, Wd, y, B)
        torch.cuda.synchronize()
        first = to_host(ys[0])
        for y in ys[1:]:
            np.testing.assert_array_equal(to_host(y), first)
        rows = np.unique(np.concatenate([np.arange(0, N, 97), np.arange(N - 200, N)]))
        ref = orc.linear(x, W[rows])
        ok, worst, idx = within_tolerance(first[:, rows], ref)
        assert ok, (worst, idx)
        g = torch.cuda.CUDAGraph()
        yg = empty_out(B, N)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            dep.dep_projection_run(plan, xd, Wd, yg, B, stream=s.cuda_stream)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            dep.dep_projection_run(plan, xd, Wd, yg, B, stream=s.cuda_stream)
        for _ in range(3):
            yg.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            np.testing.assert_array_equal(to_host(yg), first)
        assert dep.dep_projection_device_status(plan) == 0
    finally:
        dep.dep_projection_plan_destroy(plan)


@pytest.mark.parametrize("N,K", [(333, 1000), (97, 264), (1000, 3136), (700, 2048)])
@pytest.mark.parametrize("R", [32, 96, 192, 256])
def test_xm_pairs_parity_vs_oracle(dep, orc, plans, N, K, R):
    """Pairs of blocks (each half of K) on tiles of R weight rows; the same
    passes, stage widths and ragged shapes as the whole-K blocks (K = 264: five
    slices, two for rank 0 and three for rank 1); 1, 3 and all pairs of SMs
    (pairs taking several tiles in turn)."""
    plan = plans(N, K)
    for B in (17, 64, 100, 129, 300):
        x, W, ref = inputs_and_ref(orc, N, K, B)
        for cols in (128, 256):
            for tile_k in (64, 128, 256):
                st = deepest(R, tile_k, cols, pair=True)
                if not st:
                    continue
                for ctas in (2, 6, sm_count() // 2 * 2):
                    y = run(dep, plan, x, W, N, xm_tactic(dep, R, cols, tile_k, st, ctas, pair=True))
                    ok, worst, idx = within_tolerance(y, ref)
                    assert ok, (B, cols, tile_k, st, ctas, worst, idx)


@pytest.mark.parametrize("cols,B", [(128, 40), (128, 128), (256, 256), (256, 100)])
def test_xm_pairs_bits_independent_of_grid_depth_and_stage_width(dep, plans, cols, B):
    """A pair's halves are fixed (the first and second half of the 64-column
    slices) and added in that order: identical bits whatever the number of pairs,
    the ring depth and the slices per stage."""
    N, K, R = 1000, 3072, 96
    plan = plans(N, K)
    W = synth.normal_bf16(43, 1, (N, K), sigma=0.02)
    x = synth.normal_bf16(44, 2, (B, K))
    ref = run(dep, plan, x, W, N, xm_tactic(dep, R, cols, 64, deepest(R, 64, cols, pair=True), sm_count() // 2 * 2,
                                            pair=True))
    for tile_k in (64, 128, 256):
        top = deepest(R, tile_k, cols, pair=True)
        for st in sorted({2, top}) if top else ():
            for ctas in (2, 10, sm_count() // 2 * 2):
                y = run(dep, plan, x, W, N, xm_tactic(dep, R, cols, tile_k, st, ctas, pair=True))
                np.testing.assert_array_equal(y, ref, err_msg=str((tile_k, st, ctas)))


def test_xm_pairs_small_integers_exact_and_negation(dep, orc, plans):
    """Exact small-integer sums equal the oracle bit for bit; y(-x) = -y(x)."""
    rng = np.random.default_rng(47)
    N, K = 700, 2048
    x = np.vectorize(exact_bf16)(rng.integers(-8, 9, (256, K))).astype(np.uint16)
    W = np.vectorize(exact_bf16)(rng.integers(-8, 9, (N, K))).astype(np.uint16)
    plan = plans(N, K)
    ref = orc.linear(x, W)
    for R, cols, tile_k in ((192, 256, 64), (96, 128, 128), (32, 256, 64)):
        t = xm_tactic(dep, R, cols, tile_k, deepest(R, tile_k, cols, pair=True), 8, pair=True)
        np.testing.assert_array_equal(run(dep, plan, x, W, N, t), ref, err_msg=str((R, cols, tile_k)))
    xg = synth.normal_bf16(48, 2, (256, K))
    Wg = synth.normal_bf16(48, 1, (N, K), sigma=0.02)
    t = xm_tactic(dep, 192, 256, 64, deepest(192, 64, 256, pair=True), sm_count() // 2 * 2, pair=True)
    y = run(dep, plan, xg, Wg, N, t)
    yn = run(dep, plan, xg ^ np.uint16(0x8000), Wg, N, t)
    nz = synth.bf16_to_f32(y) != 0
    np.testing.assert_array_equal(yn[nz], y[nz] ^ np.uint16(0x8000))


def test_xm_pairs_default_plan_dsa_256_rows(dep, orc):
    """The default plan of the DSA input projection at 256 rows: pairs of blocks
    on 76 tiles of 192 rows; repeated runs and CUDA-graph replays give identical
    bits, within tolerance of the oracle on sampled rows."""
    N, K, B = 14560, 7168, 256
    plan = dep.dep_projection_plan(N, K, [B])
    try:
        t = dep.dep_projection_plan_query(plan, B)
        assert (t.kind, t.splits, t.tile_n) == (dep.DEP_KIND_TC_XM, 2, 192)
        W = synth.normal_bf16(49, 1, (N, K), sigma=0.02)
        x = synth.normal_bf16(50, 2, (B, K))
        xd, Wd = to_dev(x), to_dev(W)
        ys = [empty_out(B, N) for _ in range(3)]
        for y in ys:
            dep.dep_projection_run(plan, xd, Wd, y, B)
        torch.cuda.synchronize()
        first = to_host(ys[0])
        for y in ys[1:]:
            np.testing.assert_array_equal(to_host(y), first)
        rows = np.unique(np.concatenate([np.arange(0, N, 89), np.arange(N - 200, N)]))
        ok, worst, idx = within_tolerance(first[:, rows], orc.linear(x, W[rows]))
        assert ok, (worst, idx)
        g = torch.cuda.CUDAGraph()
        yg = empty_out(B, N)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            dep.dep_projection_run(plan, xd, Wd, yg, B, stream=s.cuda_stream)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            dep.dep_projection_run(plan, xd, Wd, yg, B, stream=s.cuda_stream)
        for _ in range(3):
            yg.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            np.testing.assert_array_equal(to_host(yg), first)
        assert dep.dep_projection_device_status(plan) == 0
    finally:
        dep.dep_projection_plan_destroy(plan)
