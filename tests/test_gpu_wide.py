"""The wide-batch tensor-core tactic (DEP_KIND_TC_WIDE) against the oracle.

Each block streams a group of 2 or 4 weight tiles of 128 rows against every x
slice; groups split across blocks by the stream-K ranges are reduced by the
blocks that share them (each a part of the columns), adding the blocks' FP32
partials in increasing block order.  Checked here: the acceptance tolerance
against the exact oracle at every MMA width and group size, ragged N, K and B,
grids of 1, 7 and all SMs; the split-K combination bit for bit from the
partials the blocks left; whole groups equal the one-tile stream-K kernel bit
for bit (same MMAs in the same order); exact small-integer sums; sign symmetry;
run-to-run and CUDA-graph determinism.
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

KINDS = [(32, 2), (32, 4), (64, 2), (64, 4), (128, 2), (128, 4), (256, 2)]  # (MMA width NT, tiles per group G)
SMEM_MAX = 227 * 1024


def sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


def stages_for(NT, G, tile_k, want=6):
    """Deepest ring (at most `want`) whose shared memory fits one block."""
    atom = G * 16384 + NT * 128
    for st in range(want, 1, -1):
        if 1024 + st * (tile_k // 64) * atom + (2 * st + 5 + 64) * 8 + 16 <= SMEM_MAX:
            return st
    return 0


def wide_tactic(dep, NT, G, ctas, stages, tile_k=64, max_rows=None):
    return dep.dep_tactic_t(max_rows=max_rows or NT, kind=dep.DEP_KIND_TC_WIDE, ctas=ctas, tile_n=128 * G,
                            tile_k=tile_k, stages=stages, cols=NT)


def run(dep, plan, x, W, N, tactic):
    B = x.shape[0]
    y = empty_out(B, N)
    dep.dep_projection_run_tactic(plan, tactic, to_dev(x), to_dev(W), y, B)
    torch.cuda.synchronize()
    return to_host(y)


@pytest.fixture(scope="module")
def plans(dep):
    cache = {}

    def get(N, K, flags=0):
        if (N, K, flags) not in cache:
            p = dep.dep_projection_plan(N, K, [256], flags)
            # an entry of the widest group grows the workspace for every wide tactic
            dep.dep_projection_plan_set(p, wide_tactic(dep, 256, 2, sm_count(), 3, max_rows=1 << 20))
            cache[(N, K, flags)] = p
        return cache[(N, K, flags)]

    yield get
    for p in cache.values():
        assert dep.dep_projection_device_status(p) == 0
        dep.dep_projection_plan_destroy(p)


@pytest.mark.parametrize("N,K", [(256, 64), (333, 1000), (97, 264), (1000, 3000)])
@pytest.mark.parametrize("NT,G", KINDS)
def test_wide_parity_vs_oracle(dep, orc, plans, N, K, NT, G):
    """Every MMA width and group size; 1 or 2 slices per stage; partial, full and
    multi-pass batches; grids of 1, 7 and all SMs (whole and split groups, ragged
    N and K tails, groups whose second tile lies past N)."""
    plan = plans(N, K)
    W = synth.normal_bf16(N + NT + G, 1, (N, K), sigma=0.02)
    for B in sorted({min(NT, 5), NT - 3, NT, NT + 7}):
        x = synth.normal_bf16(B + NT, 2, (B, K))
        ref = orc.linear(x, W)
        for tile_k in (64, 128):
            st = stages_for(NT, G, tile_k)
            if not st:
                continue
            for ctas in (1, 7, sm_count()):
                y = run(dep, plan, x, W, N, wide_tactic(dep, NT, G, ctas, st, tile_k))
                ok, worst, idx = within_tolerance(y, ref)
                assert ok, (B, tile_k, ctas, worst, idx)


def _contributors(t, KT, U, C):
    """Blocks whose stream-K ranges meet group t, in block order, with the slot
    each left its piece in (1: the group the block starts in, else 0)."""
    owner = lambda u: ((u + 1) * C - 1) // U  # noqa: E731
    begin = lambda c: (c * U) // C  # noqa: E731
    c0, c1 = owner(t * KT), owner(t * KT + KT - 1)
    return [(c, 1 if begin(c) // KT == t else 0) for c in range(c0, c1 + 1)]


@pytest.mark.parametrize("NT,G,B,N,K", [(256, 2, 256, 1000, 4096), (128, 2, 100, 1000, 4096),
                                        (64, 4, 64, 2000, 2048), (32, 4, 20, 700, 1536), (128, 4, 128, 1300, 3072)])
def test_wide_fixup_bitexact_from_partials(dep, plans, NT, G, B, N, K):
    """For every group split across blocks, the FP32 partials the blocks left in
    the workspace (kept whole with DEP_PLAN_KEEP_PIECES), added in increasing
    block order and rounded to BF16 (nearest, ties to even), give y bit for bit."""
    plan = plans(N, K, dep.DEP_PLAN_KEEP_PIECES)
    x = synth.normal_bf16(60 + NT, 2, (B, K))
    W = synth.normal_bf16(61 + G, 1, (N, K), sigma=0.02)
    C = sm_count()
    tile_k = 64
    y = run(dep, plan, x, W, N, wide_tactic(dep, NT, G, C, stages_for(NT, G, tile_k), tile_k))
    R, half = 128 * G, G * NT // 2
    T, KT = -(-N // R), -(-K // tile_k)
    U = T * KT
    C = min(C, U)
    ws = dep.dep_projection_plan_partials(plan, C * 2 * R * NT)
    assert ws.size == C * 2 * R * NT
    r = np.arange(R)
    g, rt = r // 128, r % 128
    q, lane = rt // 32, rt % 32
    checked = 0
    for t in range(T):
        segs = _contributors(t, KT, U, C)
        if len(segs) < 2:
            continue
        n = t * R + r
        keep = n < N
        for b in range(B):
            col = g * NT + b
            h = col // half
            e = 4 * h + (q + 2) % 4
            cl = col - h * half
            off = e * 32 * half + ((cl // 4) * 32 + lane) * 4 + cl % 4
            s = None
            for c, slot in segs:
                p = ws[(c * 2 + slot) * R * NT + off].astype(np.float32)
                s = p if s is None else (s + p).astype(np.float32)
            want = synth.bf16_from_f64(s.astype(np.float64))  # float32 -> float64 is exact
            np.testing.assert_array_equal(y[b, n[keep]], want[keep])
            checked += int(keep.sum())
    assert checked > 0


@pytest.mark.parametrize("NT,G,B", [(256, 2, 256), (128, 2, 77), (64, 4, 64), (64, 2, 40)])
def test_wide_whole_groups_equal_one_tile_kernel(dep, plans, NT, G, B):
    """With one block per group (no split) every output is its tile's TMEM
    accumulator rounded once, from the same MMAs in the same order as the
    stream-K tensor-core kernel with one block per 128-row tile: equal bits.
    (At N <= 32 the one-tile kernel splits every stage's K steps between two
    MMA issuers and adds their two accumulators at the end, which the group
    kernels do not, so the comparison is made at N >= 64.)"""
    N, K = 1500, 2048
    plan = plans(N, K)
    x = synth.normal_bf16(70, 2, (B, K))
    W = synth.normal_bf16(71, 1, (N, K), sigma=0.02)
    groups, tiles = -(-N // (128 * G)), -(-N // 128)
    y = run(dep, plan, x, W, N, wide_tactic(dep, NT, G, groups, stages_for(NT, G, 64), 64))
    one = dep.dep_tactic_t(max_rows=NT, kind=dep.DEP_KIND_TC, ctas=tiles, tile_n=128, tile_k=64,
                           stages=3 if NT == 256 else 4, cols=NT)
    np.testing.assert_array_equal(y, run(dep, plan, x, W, N, one))


def test_wide_small_integers_exact(dep, orc, plans):
    """Small-integer inputs give exact FP32 sums whatever the split: every grid
    equals the exact oracle bit for bit."""
    rng = np.random.default_rng(19)
    B, N, K = 200, 700, 2048
    x = np.vectorize(exact_bf16)(rng.integers(-8, 9, (B, K))).astype(np.uint16)
    W = np.vectorize(exact_bf16)(rng.integers(-8, 9, (N, K))).astype(np.uint16)
    plan = plans(N, K)
    ref = orc.linear(x, W)
    for NT, G in ((256, 2), (128, 4), (64, 2)):
        for ctas in (1, 3, sm_count()):
            np.testing.assert_array_equal(run(dep, plan, x, W, N, wide_tactic(dep, NT, G, ctas,
                                                                               stages_for(NT, G, 64))), ref)


def test_wide_negation_symmetric(dep, plans):
    """y(-x) = -y(x) bit for bit: every FP32 step of the split combination is
    sign-symmetric."""
    N, K, B = 900, 4096, 256
    plan = plans(N, K)
    x = synth.normal_bf16(23, 2, (B, K))
    W = synth.normal_bf16(23, 1, (N, K), sigma=0.02)
    t = wide_tactic(dep, 256, 2, sm_count(), 3)
    y = run(dep, plan, x, W, N, t)
    yn = run(dep, plan, x ^ np.uint16(0x8000), W, N, t)
    nz = synth.bf16_to_f32(y) != 0
    np.testing.assert_array_equal(yn[nz], y[nz] ^ np.uint16(0x8000))


@pytest.mark.parametrize("NT,G,B", [(256, 2, 256), (128, 2, 128), (64, 4, 48)])
def test_wide_determinism_and_graph_replay(dep, NT, G, B):
    """Repeated runs and CUDA-graph replays of a split launch give identical bits
    (the flags a launch consumes are clear for the next one)."""
    N, K = 14560, 7168
    plan = dep.dep_projection_plan(N, K, [B])
    try:
        t = wide_tactic(dep, NT, G, sm_count(), stages_for(NT, G, 64), max_rows=B)
        dep.dep_projection_plan_set(plan, t)
        x = to_dev(synth.normal_bf16(B, 2, (B, K)))
        W = to_dev(synth.normal_bf16(5, 1, (N, K), 0.02))
        ref = empty_out(B, N)
        dep.dep_projection_run(plan, x, W, ref, B)
        torch.cuda.synchronize()
        for _ in range(5):
            y = empty_out(B, N)
            dep.dep_projection_run(plan, x, W, y, B)
            torch.cuda.synchronize()
            assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
        y = empty_out(B, N)
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            dep.dep_projection_run(plan, x, W, y, B, s)
        for _ in range(3):
            y.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
        assert dep.dep_projection_device_status(plan) == 0
    finally:
        dep.dep_projection_plan_destroy(plan)


# ---------------- a thread-block cluster of k CTAs per group (DEP_KIND_TC_CLUSTER) ----------------

def cluster_stages(NT, G, k, want=5):
    """Deepest weight ring (at most `want`) that fits with two or more x stages
    and holds the peers' partials and the y staging once idle (the kernel's own
    rule).  G = 3 stands for a 128-row and a 64-row tile (192 rows)."""
    tiles = 2 if G == 3 else G
    ws, xs = (24576 if G == 3 else G * 16384), NT * 128
    half = tiles * NT // 2
    cbw = max(16, half // 8)
    ncb = half // cbw
    recv = (k - 1) * 8 * -(-ncb // k) * 32 * cbw * 4
    need = -(-recv // 1024) * 1024 + 2 * 2 * cbw * 128 * 2  # received partials, then two y staging buffers
    for sw in range(want, 1, -1):
        for sx in range(4, 1, -1):
            if 1024 + sw * ws + sx * xs + (2 * sw + 2 * sx + 16) * 8 + 16 <= SMEM_MAX:
                if need <= sw * ws + sx * xs:
                    return sw
                break
    return 0


def cluster_tactic(dep, NT, G, k, clusters, stages, max_rows=None):
    return dep.dep_tactic_t(max_rows=max_rows or NT, kind=dep.DEP_KIND_TC_CLUSTER, ctas=clusters * k,
                            tile_n=192 if G == 3 else 128 * G, tile_k=64, stages=stages, cols=NT, splits=k)


def group_rows(G):
    return 192 if G == 3 else 128 * G


CLUSTER_KINDS = KINDS + [(64, 3), (128, 3), (256, 3)]  # G = 3: a 128-row and a 64-row tile


@pytest.mark.parametrize("N,K", [(256, 64), (333, 1000), (97, 264), (1000, 3000)])
@pytest.mark.parametrize("NT,G", CLUSTER_KINDS)
def test_cluster_parity_vs_oracle(dep, orc, plans, N, K, NT, G):
    """Every MMA width and group size (two or four 128-row tiles, or a 128-row
    and a 64-row tile); clusters of 1-4 CTAs (fewer where K has fewer 64-column
    k-tiles); one cluster, 3 clusters and one per group (clusters looping over
    several groups); partial, full and multi-pass batches."""
    plan = plans(N, K)
    W = synth.normal_bf16(N + NT + G + 7, 1, (N, K), sigma=0.02)
    groups = -(-N // group_rows(G))
    for B in sorted({min(NT, 5), NT - 3, NT, NT + 7}):
        x = synth.normal_bf16(B + NT + 1, 2, (B, K))
        ref = orc.linear(x, W)
        for k in (1, 2, 3, 4):
            st = cluster_stages(NT, G, k)
            if not st:
                continue
            for clusters in sorted({1, 3, groups}):
                y = run(dep, plan, x, W, N, cluster_tactic(dep, NT, G, k, clusters, st))
                ok, worst, idx = within_tolerance(y, ref)
                assert ok, (B, k, clusters, worst, idx)


@pytest.mark.parametrize("NT,G,k,B,N,K", [(256, 2, 2, 256, 1000, 4096), (128, 2, 3, 100, 1500, 4096),
                                          (64, 4, 4, 64, 2000, 2048), (32, 2, 3, 20, 700, 1536),
                                          (128, 4, 2, 128, 1300, 3072), (256, 2, 4, 250, 600, 8192)])
def test_cluster_equals_stream_k_with_the_same_pieces(dep, plans, NT, G, k, B, N, K):
    """With T k blocks the stream-K wide kernel cuts every group into the same k
    K pieces as a cluster of k CTAs, and adds them in the same (block = rank)
    order; its fix-up is checked bit for bit from its partials above.  The two
    kernels must give identical bits."""
    plan = plans(N, K)
    x = synth.normal_bf16(80 + NT, 2, (B, K))
    W = synth.normal_bf16(81 + k, 1, (N, K), sigma=0.02)
    T = -(-N // (128 * G))
    y = run(dep, plan, x, W, N, cluster_tactic(dep, NT, G, k, T, cluster_stages(NT, G, k)))
    ref = run(dep, plan, x, W, N, wide_tactic(dep, NT, G, T * k, stages_for(NT, G, 64), 64))
    np.testing.assert_array_equal(y, ref)


@pytest.mark.parametrize("NT,G,B", [(256, 2, 256), (64, 4, 33)])
def test_cluster_one_cta_per_group_equals_one_tile_kernel(dep, plans, NT, G, B):
    """k = 1: every output is its tile's accumulator rounded once, from the same
    MMAs in the same order as the one-tile stream-K kernel with a block per tile."""
    N, K = 1500, 2048
    plan = plans(N, K)
    x = synth.normal_bf16(90, 2, (B, K))
    W = synth.normal_bf16(91, 1, (N, K), sigma=0.02)
    y = run(dep, plan, x, W, N, cluster_tactic(dep, NT, G, 1, -(-N // (128 * G)), cluster_stages(NT, G, 1)))
    one = dep.dep_tactic_t(max_rows=NT, kind=dep.DEP_KIND_TC, ctas=-(-N // 128), tile_n=128, tile_k=64,
                           stages=3 if NT == 256 else 4, cols=NT)
    np.testing.assert_array_equal(y, run(dep, plan, x, W, N, one))


def test_cluster_small_integers_exact_and_negation(dep, orc, plans):
    """Exact small-integer sums equal the oracle bit for bit for clusters of 1-4
    CTAs; y(-x) = -y(x) bit for bit."""
    rng = np.random.default_rng(29)
    B, N, K = 200, 700, 2048
    x = np.vectorize(exact_bf16)(rng.integers(-8, 9, (B, K))).astype(np.uint16)
    W = np.vectorize(exact_bf16)(rng.integers(-8, 9, (N, K))).astype(np.uint16)
    plan = plans(N, K)
    ref = orc.linear(x, W)
    for NT, G in ((256, 2), (128, 4), (256, 3)):
        for k in (1, 2, 3, 4):
            t = cluster_tactic(dep, NT, G, k, -(-N // group_rows(G)), cluster_stages(NT, G, k))
            np.testing.assert_array_equal(run(dep, plan, x, W, N, t), ref)
    xn = synth.normal_bf16(31, 2, (B, K))
    Wn = synth.normal_bf16(31, 1, (N, K), sigma=0.02)
    t = cluster_tactic(dep, 256, 2, 3, 2, cluster_stages(256, 2, 3))
    y = run(dep, plan, xn, Wn, N, t)
    yn = run(dep, plan, xn ^ np.uint16(0x8000), Wn, N, t)
    nz = synth.bf16_to_f32(y) != 0
    np.testing.assert_array_equal(yn[nz], y[nz] ^ np.uint16(0x8000))


@pytest.mark.parametrize("NT,G,k,B", [(256, 2, 2, 256), (128, 2, 2, 128), (64, 4, 4, 64), (256, 3, 2, 256)])
def test_cluster_determinism_and_graph_replay(dep, NT, G, k, B):
    """Repeated runs and CUDA-graph replays give identical bits; the bounded
    waits all complete (device status 0)."""
    N, K = 14560, 7168
    plan = dep.dep_projection_plan(N, K, [B])
    try:
        T = -(-N // group_rows(G))
        dep.dep_projection_plan_set(plan, cluster_tactic(dep, NT, G, k, T, cluster_stages(NT, G, k), max_rows=B))
        x = to_dev(synth.normal_bf16(B, 2, (B, K)))
        W = to_dev(synth.normal_bf16(5, 1, (N, K), 0.02))
        ref = empty_out(B, N)
        dep.dep_projection_run(plan, x, W, ref, B)
        torch.cuda.synchronize()
        for _ in range(5):
            y = empty_out(B, N)
            dep.dep_projection_run(plan, x, W, y, B)
            torch.cuda.synchronize()
            assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
        y = empty_out(B, N)
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            dep.dep_projection_run(plan, x, W, y, B, s)
        for _ in range(3):
            y.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
        assert dep.dep_projection_device_status(plan) == 0
    finally:
        dep.dep_projection_plan_destroy(plan)
