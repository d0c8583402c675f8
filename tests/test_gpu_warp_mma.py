"""The warp-level MMA tactic for small weights (DEP_KIND_WARP_MMA) against the oracle.

One block per tile of 16 weight rows sums the tile's whole K (or 2 or 4 blocks
of a cluster each a K piece, added in rank order in the first block) with
mma.sync (m16n8k16, BF16 in, FP32 accumulators in registers): four compute
warps take the 64-column slices g with g % 4 = warp, each in increasing K
order, and the four partials are added in warp order.  Checked here: the acceptance tolerance
against the exact oracle on ragged N, K and B (passes of 16 rows), one, two or
four slices per stage, shallow and deep rings; identical bits whatever the
stage width and the ring depth; exact small-integer sums; sign symmetry; the
default plan of o_proj at 16 rows, repeated and replayed from a CUDA graph.
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


def mma_tactic(dep, tile_k, stages, max_rows=16, splits=0):
    return dep.dep_tactic_t(max_rows=max_rows, kind=dep.DEP_KIND_WARP_MMA, ctas=1, tile_n=16, tile_k=tile_k,
                            stages=stages, cols=16, splits=splits)


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
            cache[(N, K)] = dep.dep_projection_plan(N, K, [16])
        return cache[(N, K)]

    yield get
    for p in cache.values():
        assert dep.dep_projection_device_status(p) == 0
        dep.dep_projection_plan_destroy(p)


@pytest.mark.parametrize("N,K", [(333, 1000), (97, 264), (1000, 3136), (700, 2048), (7168, 1536), (3640, 128)])
@pytest.mark.parametrize("splits", [0, 2, 4])
def test_warp_mma_parity_vs_oracle(dep, orc, plans, N, K, splits):
    """Ragged last tile (N % 16 != 0), K not a multiple of 64 (one copy per slice,
    a ragged last slice) or of the stage width (one copy per stage, the last
    stage partly past K), batches of 1, 5, 16 rows and 17, 40 (two and three
    passes); 1, 2 or 4 slices per stage, rings of 2 and 6; whole K per block or
    2 and 4 K pieces per tile in a cluster (K = 128: two slices, so four pieces
    run as two)."""
    plan = plans(N, K)
    W = synth.normal_bf16(N + K, 1, (N, K), sigma=0.02)
    for B in (1, 5, 16, 17, 40):
        x = synth.normal_bf16(N + B, 2, (B, K))
        ref = orc.linear(x, W)
        for tile_k in (64, 128, 256):
            for st in (2, 6):
                y = run(dep, plan, x, W, N, mma_tactic(dep, tile_k, st, splits=splits))
                ok, worst, idx = within_tolerance(y, ref)
                assert ok, (B, tile_k, st, worst, idx)


@pytest.mark.parametrize("B", [3, 16, 29])
@pytest.mark.parametrize("splits", [0, 2, 4])
def test_warp_mma_bits_independent_of_stage_width_and_depth(dep, plans, B, splits):
    """Slice g of a block's piece goes to compute warp g % 4 whatever the stage
    width, each warp adds its slices in K order, and the pieces are added in
    rank order: identical bits for every tile_k and ring depth at a given number
    of pieces."""
    N, K = 1000, 3136
    plan = plans(N, K)
    W = synth.normal_bf16(61, 1, (N, K), sigma=0.02)
    x = synth.normal_bf16(62, 2, (B, K))
    ref = run(dep, plan, x, W, N, mma_tactic(dep, 256, 4, splits=splits))
    for tile_k in (64, 128, 256):
        for st in (2, 3, 8):
            np.testing.assert_array_equal(run(dep, plan, x, W, N, mma_tactic(dep, tile_k, st, splits=splits)), ref,
                                          err_msg=str((tile_k, st)))


def test_warp_mma_small_integers_exact_and_negation(dep, orc, plans):
    """Exact small-integer sums equal the oracle bit for bit; y(-x) = -y(x)."""
    rng = np.random.default_rng(67)
    N, K = 700, 2048
    x = np.vectorize(exact_bf16)(rng.integers(-8, 9, (16, K))).astype(np.uint16)
    W = np.vectorize(exact_bf16)(rng.integers(-8, 9, (N, K))).astype(np.uint16)
    plan = plans(N, K)
    for splits in (0, 2, 4):
        np.testing.assert_array_equal(run(dep, plan, x, W, N, mma_tactic(dep, 256, 4, splits=splits)),
                                      orc.linear(x, W))
    xg = synth.normal_bf16(68, 2, (16, K))
    Wg = synth.normal_bf16(68, 1, (N, K), sigma=0.02)
    t = mma_tactic(dep, 128, 4)
    y = run(dep, plan, xg, Wg, N, t)
    yn = run(dep, plan, xg ^ np.uint16(0x8000), Wg, N, t)
    nz = synth.bf16_to_f32(y) != 0
    np.testing.assert_array_equal(yn[nz], y[nz] ^ np.uint16(0x8000))


@pytest.mark.parametrize("B", [8, 16])
def test_warp_mma_default_plan_oproj(dep, orc, B):
    """The default plan of o_proj (7168 x 12288) takes this kind at 8 and 16
    rows; repeated runs and CUDA-graph replays give identical bits, within
    tolerance of the oracle on sampled rows."""
    N, K = 7168, 12288
    plan = dep.dep_projection_plan(N, K, [B])
    try:
        assert dep.dep_projection_plan_query(plan, B).kind == dep.DEP_KIND_WARP_MMA
        W = synth.normal_bf16(71, 1, (N, K), sigma=0.02)
        x = synth.normal_bf16(72, 2, (B, K))
        xd, Wd = to_dev(x), to_dev(W)
        ys = [empty_out(B, N) for _ in range(3)]
        for y in ys:
            dep.dep_projection_run(plan, xd, Wd, y, B)
        torch.cuda.synchronize()
        first = to_host(ys[0])
        for y in ys[1:]:
            np.testing.assert_array_equal(to_host(y), first)
        rows = np.unique(np.concatenate([np.arange(0, N, 37), np.arange(N - 40, N)]))
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
