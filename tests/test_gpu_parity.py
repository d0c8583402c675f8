"""GPU parity of the decode projection against the CPU oracle and the FP32 mirror.

Every case calls the CUDA path through the C ABI (the ctypes binding) and
compares element by element: against the exact oracle within the acceptance
tolerance |y - y_ref| <= 2^-7 |y_ref| + 1e-3 rms(y_ref), and -- for the split-K
FMA tactic, whose summation order is fixed and restated in oracle/mirror.c --
against the FP32 mirror bit for bit.
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


def fma_tactic(dep, cols, ctas, stages=None, max_rows=None, tile_n=32):
    return dep.dep_tactic_t(max_rows=max_rows or cols, kind=dep.DEP_KIND_SPLITK_FMA, ctas=ctas,
                            tile_n=tile_n, tile_k=256, stages=stages or (6 if cols >= 8 else 4),
                            cols=cols)


@pytest.fixture(scope="module")
def plan_cache(dep):
    plans = {}
    yield plans
    for p in plans.values():
        dep.dep_projection_plan_destroy(p)


def get_plan(dep, cache, N, K, batches=(1, 2, 4, 8, 16, 32, 64, 128, 256)):
    key = (N, K, tuple(batches))
    if key not in cache:
        cache[key] = dep.dep_projection_plan(N, K, list(batches))
    return cache[key]


def run(dep, plan, x, W, N, tactic=None):
    xd, Wd = to_dev(x), to_dev(W)
    y = empty_out(x.shape[0], N)
    if tactic is None:
        dep.dep_projection_run(plan, xd, Wd, y, x.shape[0])
    else:
        dep.dep_projection_run_tactic(plan, tactic, xd, Wd, y, x.shape[0])
    torch.cuda.synchronize()
    return to_host(y)


def test_bounded_wait_gives_up_and_reports(dep):
    """A wait that can never be satisfied returns by itself with its code."""
    assert dep.dep_projection_selftest_timeout(2000) == dep.DEP_DEV_TIMEOUT_CONSUMER
    # the context is still usable afterwards
    a = torch.ones(4, device="cuda")
    assert float(a.sum()) == 4.0


# shapes spanning several tiles plus ragged tails in N (tile 32/64) and K (tile 256)
SHAPES = [(333, 3000), (64, 256), (97, 264), (1, 8), (1000, 1032)]


@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("cols,tile_n", [(1, 32), (1, 64), (2, 32), (2, 64), (4, 32), (4, 64), (8, 32)])
@pytest.mark.parametrize("ctas", [1, 7, 152, 1000])
def test_fma_bitexact_vs_mirror(dep, orc, plan_cache, N, K, cols, tile_n, ctas):
    B = {1: 1, 2: 2, 4: 3, 8: 8}[cols]
    x = synth.normal_bf16(N + cols, 2, (B, K))
    W = synth.normal_bf16(N + ctas, 1, (N, K), sigma=0.02)
    t = fma_tactic(dep, cols, ctas, tile_n=tile_n)
    y = run(dep, get_plan(dep, plan_cache, N, K), x, W, N, t)
    T = -(-N // t.tile_n) * -(-K // 256)
    want = orc.mirror_fma(x, W, min(ctas, T), t.tile_n)
    np.testing.assert_array_equal(y, want)
    ok, worst, idx = within_tolerance(y, orc.linear(x, W))
    assert ok, (worst, idx)


@pytest.mark.parametrize("B", list(range(1, 18)) + [31, 33, 64, 100, 256, 300])
def test_default_plan_any_batch(dep, orc, plan_cache, B):
    """Any B >= 1 works through the binning rule (wide batches run in passes)."""
    N, K = 200, 1280
    x = synth.normal_bf16(B, 2, (B, K))
    W = synth.normal_bf16(77, 1, (N, K), sigma=0.02)
    plan = get_plan(dep, plan_cache, N, K)
    y = run(dep, plan, x, W, N)
    ok, worst, idx = within_tolerance(y, orc.linear(x, W))
    assert ok, (worst, idx)
    t = dep.dep_projection_plan_query(plan, B)
    if t.kind == dep.DEP_KIND_SPLITK_FMA:
        T = -(-N // t.tile_n) * -(-K // 256)
        np.testing.assert_array_equal(y, orc.mirror_fma(x, W, min(t.ctas, T), t.tile_n))


def test_small_integers_exact(dep, orc, plan_cache):
    """Small-integer inputs: all partial sums are exact in FP32, so the GPU must
    equal the exact oracle bit for bit whatever its order."""
    rng = np.random.default_rng(5)
    B, N, K = 16, 300, 2048
    xi, wi = rng.integers(-8, 9, (B, K)), rng.integers(-8, 9, (N, K))
    x = np.vectorize(exact_bf16)(xi).astype(np.uint16)
    W = np.vectorize(exact_bf16)(wi).astype(np.uint16)
    want = orc.linear(x, W)
    np.testing.assert_array_equal(want, synth.bf16_from_f64((xi @ wi.T).astype(np.float64)))
    np.testing.assert_array_equal(run(dep, get_plan(dep, plan_cache, N, K), x, W, N), want)


def test_closed_forms(dep, orc, plan_cache):
    """Identity-like W returns x; all-ones x returns BF16 row sums (oracle)."""
    N, K = 128, 512
    x = synth.normal_bf16(1, 2, (4, K))
    W = np.zeros((N, K), dtype=np.uint16)
    W[np.arange(N), np.arange(N)] = 0x3F80
    y = run(dep, get_plan(dep, plan_cache, N, K), x, W, N)
    xz = x[:, :N].copy()
    xz[synth.bf16_to_f32(xz) == 0] = 0
    np.testing.assert_array_equal(y, xz)
    W = synth.normal_bf16(2, 1, (N, K), sigma=0.02)
    ones = np.full((2, K), 0x3F80, dtype=np.uint16)
    ok, worst, idx = within_tolerance(run(dep, get_plan(dep, plan_cache, N, K), ones, W, N),
                                      orc.linear(ones, W))
    assert ok, (worst, idx)


def test_invariants_bitwise(dep, plan_cache):
    """Negating x negates y and scaling x by 2^3 scales y: bit for bit, since
    every FP32 step commutes with both."""
    N, K = 500, 4096
    x = synth.normal_bf16(3, 2, (4, K))
    W = synth.normal_bf16(3, 1, (N, K), sigma=0.02)
    plan = get_plan(dep, plan_cache, N, K)
    y = run(dep, plan, x, W, N)
    yn = run(dep, plan, x ^ np.uint16(0x8000), W, N)
    nz = synth.bf16_to_f32(y) != 0
    np.testing.assert_array_equal(yn[nz], y[nz] ^ np.uint16(0x8000))
    f = synth.bf16_to_f32(x)
    x8 = np.where(f != 0, x + np.uint16(3 << 7), x).astype(np.uint16)
    y8 = run(dep, plan, x8, W, N)
    np.testing.assert_array_equal(y8[nz], (y[nz] + np.uint16(3 << 7)).astype(np.uint16))


def test_row_permutation_within_tiles(dep, plan_cache):
    """An output's summation order depends only on its row tile and k, so
    permuting W's rows inside aligned blocks of 32 (a whole number of rows of
    every tile size) permutes y's columns bit for bit."""
    N, K = 256, 2048
    x = synth.normal_bf16(4, 2, (2, K))
    W = synth.normal_bf16(4, 1, (N, K), sigma=0.02)
    plan = get_plan(dep, plan_cache, N, K)
    y = run(dep, plan, x, W, N)
    rng = np.random.default_rng(0)
    perm = np.concatenate([32 * j + rng.permutation(32) for j in range(N // 32)])
    np.testing.assert_array_equal(run(dep, plan, x, W[perm], N), y[:, perm])


def test_determinism_repeated_and_concurrent(dep, plan_cache):
    """The same call gives the same bits every time, also with other streams busy."""
    N, K, B = 7168, 4096, 4
    x, W = to_dev(synth.normal_bf16(8, 2, (B, K))), to_dev(synth.normal_bf16(8, 1, (N, K), 0.02))
    plan = get_plan(dep, plan_cache, N, K)
    ref = empty_out(B, N)
    dep.dep_projection_run(plan, x, W, ref, B)
    torch.cuda.synchronize()
    other = torch.cuda.Stream()
    big = torch.randn(4096, 4096, device="cuda")
    for i in range(30):
        y = empty_out(B, N)
        if i % 3 == 0:
            with torch.cuda.stream(other):
                big = big @ big * 1e-3
        dep.dep_projection_run(plan, x, W, y, B)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16)), i


def test_cuda_graph_capture_and_replay(dep, plan_cache):
    """run() allocates nothing and synchronises nothing: it captures into a CUDA
    graph, and replays give the eager result (counters reset themselves)."""
    N, K, B = 1000, 3000, 4
    x, W = to_dev(synth.normal_bf16(9, 2, (B, K))), to_dev(synth.normal_bf16(9, 1, (N, K), 0.02))
    plan = get_plan(dep, plan_cache, N, K)
    eager = empty_out(B, N)
    dep.dep_projection_run(plan, x, W, eager, B)
    torch.cuda.synchronize()
    y = empty_out(B, N)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dep.dep_projection_run(plan, x, W, y, B, s)
    for _ in range(5):
        y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), eager.view(torch.int16))


def test_zero_batch_and_guard_bands(dep, plan_cache):
    """B == 0 writes nothing; a normal call writes exactly y and nothing around it."""
    N, K, B = 777, 1024, 3
    plan = get_plan(dep, plan_cache, N, K)
    x, W = to_dev(synth.normal_bf16(1, 2, (B, K))), to_dev(synth.normal_bf16(1, 1, (N, K), 0.02))
    pad = 4096
    buf = torch.full((pad + B * N + pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    y = buf[pad:pad + B * N].view(B, N)
    dep.dep_projection_run(plan, x, W, y, 0)
    torch.cuda.synchronize()
    assert bool((buf == 7.0).all())
    dep.dep_projection_run(plan, x, W, y, B)
    torch.cuda.synchronize()
    assert bool((buf[:pad] == 7.0).all()) and bool((buf[pad + B * N:] == 7.0).all())
    assert not bool((y == 7.0).all())


def test_argument_errors_on_device(dep, plan_cache):
    N, K = 64, 64
    plan = get_plan(dep, plan_cache, N, K)
    x = torch.zeros(2, K, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(N, K, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(2, N, dtype=torch.bfloat16, device="cuda")
    cases = [
        (lambda: dep.dep_projection_run(plan, x, W, y, -1), dep.DEP_ERR_INVALID_ARG),
        (lambda: dep.dep_projection_run(plan, 0, W, y, 2), dep.DEP_ERR_INVALID_ARG),
        (lambda: dep.dep_projection_run(plan, x.data_ptr() + 2, W, y, 2), dep.DEP_ERR_MISALIGNED),
        (lambda: dep.dep_projection_run(plan, x, W, W.data_ptr(), 2), dep.DEP_ERR_INVALID_ARG),
        (lambda: dep.dep_projection_run(plan, x, W, x.data_ptr(), 1), dep.DEP_ERR_INVALID_ARG),
    ]
    for fn, status in cases:
        with pytest.raises(dep.DepError) as e:
            fn()
        assert e.value.status == status
    assert dep.dep_projection_device_status(plan) == 0
    # a grid whose split-K partials exceed the plan's workspace is refused
    N, K = 7168, 12288
    big = get_plan(dep, plan_cache, N, K, (1, 2, 4, 8, 16))
    x = torch.zeros(2, K, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(N, K, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(2, N, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dep.DepError) as e:
        dep.dep_projection_run_tactic(big, fma_tactic(dep, 8, 10 ** 6), x, W, y, 2)
    assert e.value.status == dep.DEP_ERR_INVALID_ARG


@pytest.mark.parametrize("B,N", [(5, 640), (1, 333), (16, 7168), (40, 1001), (255, 14561)])
@pytest.mark.parametrize("memory", ["pinned", "pageable", "pinned-copy", "pinned-stage"])
def test_run_host_end_to_end(dep, orc, plan_cache, monkeypatch, B, N, memory):
    """The host-buffer entry point gives the device entry point's bits: pinned
    buffers through the zero-copy gather, y stored by the projection or (the
    cluster kind at B = 40, the x-on-M kind at B = 255; every kind under
    DEP_STAGING=stage) copied back by the staging kernel, chained by
    programmatic dependent launch (N odd included: a 2-byte tail; B = 255: a
    7.4 MB y, several rounds of four 16-byte vectors per copying thread),
    pageable buffers and DEP_STAGING=copy through memcpys.  Ten calls back to
    back, one sync."""
    K = 2048
    plan = get_plan(dep, plan_cache, N, K)
    if memory == "pinned-copy":
        monkeypatch.setenv("DEP_STAGING", "copy")
    if memory == "pinned-stage":
        monkeypatch.setenv("DEP_STAGING", "stage")
    xs = [synth.normal_bf16(2 + i, 2, (B, K)) for i in range(10)]
    W = synth.normal_bf16(2, 1, (N, K), sigma=0.02)
    Wd = to_dev(W)
    if memory == "pageable":
        xh = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16) for x in xs]
        yh = [torch.full((B, N), float("nan"), dtype=torch.bfloat16) for _ in xs]
    else:
        xh = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory() for x in xs]
        yh = [torch.full((B, N), float("nan"), dtype=torch.bfloat16).pin_memory() for _ in xs]
    for i in range(len(xs)):
        dep.dep_projection_run_host(plan, xh[i], Wd, yh[i], B)
    torch.cuda.synchronize()
    for x, y in zip(xs, yh):
        np.testing.assert_array_equal(y.view(torch.int16).numpy().view(np.uint16), run(dep, plan, x, W, N))
    assert dep.dep_projection_device_status(plan) == 0


@pytest.mark.parametrize("B", [4, 16, 64])
def test_run_host_chain_through_pinned_buffers(dep, plan_cache, B):
    """Calls chained through the host buffers with no synchronisation between
    them: each call's pinned output is the next call's pinned input.  The
    zero-copy gather of a call, launched with the programmatic attribute, must
    still see the y of the call before it, stored into the pinned buffer by the
    projection itself (B = 4, 16) or copied back by the staging kernel (B = 64,
    the cluster kind); it reads only after the preceding grid has completed.
    The chain gives the bits of the same chain run one synchronised call at a
    time."""
    N = K = 2048
    plan = get_plan(dep, plan_cache, N, K)
    W = synth.normal_bf16(130, 1, (N, K), sigma=0.02)
    Wd = to_dev(W)
    bufs = [torch.empty((B, K), dtype=torch.bfloat16).pin_memory() for _ in range(7)]
    bufs[0].copy_(torch.from_numpy(synth.normal_bf16(131, 2, (B, K)).view(np.int16)).view(torch.bfloat16))
    for i in range(6):
        dep.dep_projection_run_host(plan, bufs[i], Wd, bufs[i + 1], B)
    torch.cuda.synchronize()
    x = bufs[0].view(torch.int16).numpy().view(np.uint16).copy()
    for i in range(6):
        x = run(dep, plan, x, W, N)
        np.testing.assert_array_equal(bufs[i + 1].view(torch.int16).numpy().view(np.uint16), x)
    assert dep.dep_projection_device_status(plan) == 0


def test_run_host_captured_in_a_graph(dep, plan_cache):
    """The host-buffer entry point with pinned buffers inside a CUDA graph: the
    zero-copy gather and the projection that stores y into the pinned buffer
    (chained by programmatic dependent launch) replay with new inputs written
    into the same pinned buffers, and every replay gives the device entry
    point's bits."""
    N, K, B = 7168, 4096, 8
    plan = get_plan(dep, plan_cache, N, K)
    W = synth.normal_bf16(120, 1, (N, K), sigma=0.02)
    Wd = to_dev(W)
    xh = torch.empty((B, K), dtype=torch.bfloat16).pin_memory()
    yh = torch.empty((B, N), dtype=torch.bfloat16).pin_memory()
    stream = torch.cuda.Stream()
    xh.copy_(torch.from_numpy(synth.normal_bf16(121, 2, (B, K)).view(np.int16)).view(torch.bfloat16))
    with torch.cuda.stream(stream):
        dep.dep_projection_run_host(plan, xh, Wd, yh, B, stream)  # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        dep.dep_projection_run_host(plan, xh, Wd, yh, B, stream)
    for i in range(3):
        x = synth.normal_bf16(122 + i, 2, (B, K))
        xh.copy_(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16))
        yh.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(yh.view(torch.int16).numpy().view(np.uint16), run(dep, plan, x, W, N))
    assert dep.dep_projection_device_status(plan) == 0


def test_plan_save_load_roundtrip(dep, plan_cache, tmp_path):
    N, K = 7168, 12288
    plan = get_plan(dep, plan_cache, N, K, (1, 2, 4, 8, 16))
    path = str(tmp_path / "plan.txt")
    dep.dep_projection_plan_save(plan, path)
    p2 = dep.dep_projection_plan_load(path, N, K)
    try:
        assert [t.as_dict() for t in dep.dep_projection_plan_table(p2)] == \
               [t.as_dict() for t in dep.dep_projection_plan_table(plan)]
        with pytest.raises(dep.DepError) as e:
            dep.dep_projection_plan_load(path, N, K + 8)
        assert e.value.status == dep.DEP_ERR_INVALID_ARG
    finally:
        dep.dep_projection_plan_destroy(p2)


def test_stock_gemm_within_tolerance_of_oracle(orc):
    """Context: torch.mm (the stock path the pages fall back to) sits within the
    same tolerance of the oracle."""
    N, K, B = 512, 7168, 16
    x = synth.normal_bf16(6, 2, (B, K))
    W = synth.normal_bf16(6, 1, (N, K), sigma=0.02)
    y = to_host(torch.mm(to_dev(x), to_dev(W).t()))
    ok, worst, idx = within_tolerance(y, orc.linear(x, W))
    assert ok, (worst, idx)


# ---------------- tensor-core (tcgen05) tactic ----------------

def tc_tactic(dep, NT, ctas, stages=4, tile_k=64):
    return dep.dep_tactic_t(max_rows=NT, kind=dep.DEP_KIND_TC, ctas=ctas, tile_n=128, tile_k=tile_k,
                            stages=stages, cols=NT)


SMS = None


def sm_count():
    global SMS
    if SMS is None:
        SMS = torch.cuda.get_device_properties(0).multi_processor_count
    return SMS


@pytest.mark.parametrize("N,K", [(128, 64), (333, 1000), (97, 264), (1000, 3000)])
@pytest.mark.parametrize("NT,tile_k", [(16, 64), (16, 128), (16, 256), (32, 64), (32, 256), (64, 64),
                                       (64, 128), (128, 64), (128, 128), (256, 64)])
def test_tc_parity_vs_oracle(dep, orc, plan_cache, N, K, NT, tile_k):
    """tcgen05 kernel, every MMA width, 1, 2 or 4 slices of 64 columns per stage,
    partial and full batches, stream-K grids of 1, 7 and all SMs (split tiles,
    ragged N and K tails)."""
    plan = get_plan(dep, plan_cache, N, K, (256,))
    W = synth.normal_bf16(N + NT, 1, (N, K), sigma=0.02)
    stages = {64: 4 if NT < 256 else 3, 128: 2 if NT >= 128 else 3, 256: 2}[tile_k]
    for B in sorted({1, min(NT, 5), NT}):
        x = synth.normal_bf16(B + NT, 2, (B, K))
        ref = orc.linear(x, W)
        for ctas in (1, 7, sm_count()):
            y = run(dep, plan, x, W, N, tc_tactic(dep, NT, ctas, stages, tile_k))
            ok, worst, idx = within_tolerance(y, ref)
            assert ok, (B, ctas, worst, idx)
    assert dep.dep_projection_device_status(plan) == 0


@pytest.mark.parametrize("B", [4, 16, 64])
@pytest.mark.parametrize("which", ["default", "stream-k"])
def test_tc_determinism_and_graph_replay(dep, plan_cache, B, which):
    """The tensor-core kernels' split-K combinations are order-fixed: repeated
    runs and CUDA-graph replays give identical bits (the default plan takes the
    K-piece kernel for this weight at 4 rows, warp-level MMAs on its 448 tiles of
    16 rows at 16, and x on the MMA's M side at 64 rows; the stream-K kernel is
    installed explicitly)."""
    N, K = 7168, 4096
    x, W = to_dev(synth.normal_bf16(B, 2, (B, K))), to_dev(synth.normal_bf16(5, 1, (N, K), 0.02))
    if which == "default":
        plan = get_plan(dep, plan_cache, N, K)
        want = {4: dep.DEP_KIND_TC_SPLIT, 16: dep.DEP_KIND_WARP_MMA, 64: dep.DEP_KIND_TC_XM}[B]
        assert dep.dep_projection_plan_query(plan, B).kind == want
    else:
        plan = get_plan(dep, plan_cache, N, K, (B,))
        NT = max(16, 1 << (B - 1).bit_length())
        t = tc_tactic(dep, NT, sm_count(), 3, 128)
        t.max_rows = B
        dep.dep_projection_plan_set(plan, t)
        assert dep.dep_projection_plan_query(plan, B).kind == dep.DEP_KIND_TC
    ref = empty_out(B, N)
    dep.dep_projection_run(plan, x, W, ref, B)
    torch.cuda.synchronize()
    for _ in range(10):
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


def test_tc_small_integers_exact(dep, orc, plan_cache):
    """Small-integer inputs give exact FP32 sums: the tensor-core path must equal
    the exact oracle bit for bit."""
    rng = np.random.default_rng(9)
    B, N, K = 24, 300, 2048
    xi, wi = rng.integers(-8, 9, (B, K)), rng.integers(-8, 9, (N, K))
    x = np.vectorize(exact_bf16)(xi).astype(np.uint16)
    W = np.vectorize(exact_bf16)(wi).astype(np.uint16)
    plan = get_plan(dep, plan_cache, N, K)
    assert dep.dep_projection_plan_query(plan, B).kind == dep.DEP_KIND_TC
    ref = orc.linear(x, W)
    np.testing.assert_array_equal(run(dep, plan, x, W, N), ref)
    for ctas in (1, 2, sm_count()):  # the stream-K kernel, split tiles included
        np.testing.assert_array_equal(run(dep, plan, x, W, N, tc_tactic(dep, 32, ctas, 3, 128)), ref)
    pieces = tcs_plan(dep, N, K, [tcs_tactic(dep, 32, sm_count(), s, 3, 128, max_rows=300 + s, tile_n=bm)
                                  for s in (1, 5) for bm in (64, 128)])
    try:  # the K-piece kernel, one and five pieces, 64- and 128-row tiles
        for s in (1, 5):
            for bm in (64, 128):
                y = run(dep, pieces, x, W, N, tcs_tactic(dep, 32, sm_count(), s, 3, 128, tile_n=bm))
                np.testing.assert_array_equal(y, ref)
    finally:
        dep.dep_projection_plan_destroy(pieces)


def test_tc_negation_symmetric(dep, plan_cache):
    """Negating x negates every product, and every FP32 step of the fix-up is
    sign-symmetric: y(-x) = -y(x) bit for bit on the tensor-core path too."""
    N, K, B = 500, 4096, 16
    x = synth.normal_bf16(13, 2, (B, K))
    W = synth.normal_bf16(13, 1, (N, K), sigma=0.02)
    plan = get_plan(dep, plan_cache, N, K)
    y = run(dep, plan, x, W, N)
    yn = run(dep, plan, x ^ np.uint16(0x8000), W, N)
    nz = synth.bf16_to_f32(y) != 0
    np.testing.assert_array_equal(yn[nz], y[nz] ^ np.uint16(0x8000))


def test_tuned_plan_is_valid_and_correct(dep, orc):
    """DEP_PLAN_TUNE measures candidates and keeps one per batch; the result is
    a valid table whose runs match the oracle."""
    N, K = 1000, 2048
    plan = dep.dep_projection_plan(N, K, [1, 8, 32], dep.DEP_PLAN_TUNE)
    try:
        table = dep.dep_projection_plan_table(plan)
        assert [t.max_rows for t in table] == [1, 8, 32]
        for B in (1, 8, 32):
            x = synth.normal_bf16(B, 2, (B, K))
            W = synth.normal_bf16(3, 1, (N, K), sigma=0.02)
            ok, worst, idx = within_tolerance(run(dep, plan, x, W, N), orc.linear(x, W))
            assert ok, (B, worst, idx)
    finally:
        dep.dep_projection_plan_destroy(plan)


@pytest.mark.parametrize("B,N,kind", [(2, 2048, None), (8, 2048, None), (40, 2048, None), (16, 7168, "warp"),
                                       (64, 7168, "xm"), (128, 7168, "xm-pairs")])
def test_pdl_chain_respects_data_dependencies(dep, B, N, kind):
    """With DEP_PLAN_PDL each kernel streams its first weight tiles before the
    preceding kernel finishes, but reads x only after it: a chain where every
    call's output is the next call's input (kernels back to back, outputs
    allocated beforehand) gives exactly the bits of the same chain without
    overlap -- eagerly and replayed from a CUDA graph.  At 7168 x 7168 the warp
    MMA kind serves 16 rows (its blocks of consecutive calls share SMs), the x-on-M
    kind 64 rows with whole K per block and 128 rows in pairs of blocks, whose
    epilogue exchanges partials inside each cluster."""
    K = N
    Ws = [to_dev(synth.normal_bf16(20 + i, 1, (N, K), sigma=0.02)) for i in range(6)]
    x0 = to_dev(synth.normal_bf16(20, 2, (B, K)))
    plain = dep.dep_projection_plan(N, K, [B])
    pdl = dep.dep_projection_plan(N, K, [B], dep.DEP_PLAN_PDL)
    try:
        t = dep.dep_projection_plan_query(pdl, B)
        if kind == "warp":
            assert t.kind == dep.DEP_KIND_WARP_MMA
        elif kind is not None:
            assert (t.kind, t.splits) == (dep.DEP_KIND_TC_XM, 2 if kind == "xm-pairs" else 0)
        def chain(plan, outs, stream=None):
            x = x0
            for W, y in zip(Ws, outs):
                dep.dep_projection_run(plan, x, W, y, B, stream)
                x = y

        ref = [empty_out(B, N) for _ in Ws]
        chain(plain, ref)
        got = [empty_out(B, N) for _ in Ws]
        torch.cuda.synchronize()
        chain(pdl, got)
        torch.cuda.synchronize()
        for r, g in zip(ref, got):
            assert torch.equal(r.view(torch.int16), g.view(torch.int16))
        outs = [empty_out(B, N) for _ in Ws]
        s = torch.cuda.Stream()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            chain(pdl, outs, s)
        for _ in range(3):
            for o in outs:
                o.fill_(float("nan"))
            torch.cuda.synchronize()
            graph.replay()
            torch.cuda.synchronize()
            for r, g in zip(ref, outs):
                assert torch.equal(r.view(torch.int16), g.view(torch.int16))
        assert dep.dep_projection_device_status(pdl) == 0
    finally:
        dep.dep_projection_plan_destroy(plain)
        dep.dep_projection_plan_destroy(pdl)


def test_host_fault_injection(dep, monkeypatch):
    """Failures are made on the host (no GPU fault): a forced allocation failure
    gives DEP_ERR_OOM and no plan; a forced launch failure gives DEP_ERR_CUDA
    and launches nothing; clearing the switch restores normal runs."""
    monkeypatch.setenv("DEP_FAULT", "alloc")
    with pytest.raises(dep.DepError) as e:
        dep.dep_projection_plan(256, 512, [1, 16])
    assert e.value.status == dep.DEP_ERR_OOM
    monkeypatch.setenv("DEP_FAULT", "launch")
    plan = dep.dep_projection_plan(256, 512, [1, 16])
    try:
        x = torch.ones(4, 512, dtype=torch.bfloat16, device="cuda")
        W = torch.ones(256, 512, dtype=torch.bfloat16, device="cuda")
        y = torch.full((4, 256), 7.0, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(dep.DepError) as e:
            dep.dep_projection_run(plan, x, W, y, 4)
        assert e.value.status == dep.DEP_ERR_CUDA
        torch.cuda.synchronize()
        assert bool((y == 7.0).all())
    finally:
        dep.dep_projection_plan_destroy(plan)
    monkeypatch.delenv("DEP_FAULT")
    plan = dep.dep_projection_plan(256, 512, [1, 16])
    try:
        dep.dep_projection_run(plan, x, W, y, 4)
        torch.cuda.synchronize()
        assert bool((y == 512.0).all())
    finally:
        dep.dep_projection_plan_destroy(plan)


def test_plan_file_for_another_gpu_is_refused(dep, tmp_path):
    """A table tuned on a GPU with another SM count is not applied here."""
    path = tmp_path / "other.txt"
    path.write_text("dep_projection_plan 1\ndevice other\nsms 999\nshape 256 512\nentries 1\n"
                    "1 1 999 64 256 4 1\n")
    with pytest.raises(dep.DepError) as e:
        dep.dep_projection_plan_load(str(path), 256, 512)
    assert e.value.status == dep.DEP_ERR_UNSUPPORTED


# ---------------- whole-row tactic (no cross-block split) ----------------

def rows_tactic(dep, cols, tile_n, tile_k, stages, ctas):
    return dep.dep_tactic_t(max_rows=cols, kind=dep.DEP_KIND_ROWS, ctas=ctas, tile_n=tile_n,
                            tile_k=tile_k, stages=stages, cols=cols)


def rows_fits(cols, tile_n, tile_k, stages, K):
    """Shared memory of the whole-row kernel: x (padded to 256 columns) + ring + barriers."""
    kpad = -(-K // 256) * 256
    return cols * kpad * 2 + stages * tile_n * tile_k * 2 + (3 * stages + 1) * 8 <= 227 * 1024


@pytest.mark.parametrize("N,K", [(333, 3000), (64, 256), (97, 264), (1, 8), (1000, 1032), (130, 4104)])
@pytest.mark.parametrize("cols,tile_n", [(1, 8), (1, 16), (2, 8), (2, 16), (4, 8), (4, 16)])
@pytest.mark.parametrize("tile_k,stages", [(1024, 2), (2048, 3), (4096, 2)])
def test_rows_bitexact_vs_mirror(dep, orc, plan_cache, N, K, cols, tile_n, tile_k, stages):
    """Every output is summed by one warp over all of K, whatever block takes its
    tile: the result equals the mirror's order for a tile owned whole (a grid of
    one block), bit for bit, for grids of 1, 7 and 152 blocks and more blocks
    than tiles."""
    if not rows_fits(cols, tile_n, tile_k, stages, K):
        pytest.skip("ring and x exceed shared memory")
    B = {1: 1, 2: 2, 4: 3}[cols]
    x = synth.normal_bf16(N + cols + tile_n, 2, (B, K))
    W = synth.normal_bf16(N + tile_k, 1, (N, K), sigma=0.02)
    plan = get_plan(dep, plan_cache, N, K)
    want = orc.mirror_fma(x, W, 1, 64)
    for ctas in (1, 7, 152, 1000):
        y = run(dep, plan, x, W, N, rows_tactic(dep, cols, tile_n, tile_k, stages, ctas))
        np.testing.assert_array_equal(y, want)
    assert dep.dep_projection_device_status(plan) == 0


def test_rows_wide_batch_and_oracle(dep, orc, plan_cache):
    """B larger than the tactic's x rows runs in passes; within tolerance of the oracle."""
    N, K, B = 777, 2048, 11
    x = synth.normal_bf16(31, 2, (B, K))
    W = synth.normal_bf16(31, 1, (N, K), sigma=0.02)
    y = run(dep, get_plan(dep, plan_cache, N, K), x, W, N, rows_tactic(dep, 4, 16, 2048, 3, 152))
    np.testing.assert_array_equal(y, orc.mirror_fma(x, W, 1, 64))
    ok, worst, idx = within_tolerance(y, orc.linear(x, W))
    assert ok, (worst, idx)


def test_rows_refuses_when_x_does_not_fit(dep):
    """x stays in shared memory: a K too long for it is refused, not run."""
    N, K = 8, 65536
    plan = dep.dep_projection_plan(N, K, [4])
    try:
        x = torch.zeros(4, K, dtype=torch.bfloat16, device="cuda")
        W = torch.zeros(N, K, dtype=torch.bfloat16, device="cuda")
        y = torch.zeros(4, N, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(dep.DepError) as e:
            dep.dep_projection_run_tactic(plan, rows_tactic(dep, 4, 8, 2048, 2, 152), x, W, y, 4)
        assert e.value.status == dep.DEP_ERR_UNSUPPORTED
    finally:
        dep.dep_projection_plan_destroy(plan)


def _stream_k_segments(U, C, KT, t):
    """Blocks whose ranges meet tile t's units, in block order, and the exchange slot
    each left its piece in (stream-K split): 0 = published, 1 = the reducer's own."""
    owner = lambda u: ((u + 1) * C - 1) // U  # noqa: E731
    c0, c1 = owner(t * KT), owner(t * KT + KT - 1)
    return [(c, 1 if c == c1 else 0) for c in range(c0, c1 + 1)]


@pytest.mark.parametrize("NT,B,tile_k", [(16, 16, 256), (16, 5, 64), (32, 24, 128), (64, 64, 128)])
def test_tc_fixup_bitexact_from_partials(dep, plan_cache, NT, B, tile_k):
    """The tensor cores' own summation order is not documented, but the split-K
    combination is the library's: for every tile split across blocks, the FP32
    partials the blocks left in their exchange words, added in increasing block
    order and rounded to BF16 (nearest, ties to even), give y bit for bit; every
    "full" flag is clear once the launch has finished."""
    N, K = 1000, 4096
    plan = get_plan(dep, plan_cache, N, K, (256,))
    x = synth.normal_bf16(40 + NT, 2, (B, K))
    W = synth.normal_bf16(41, 1, (N, K), sigma=0.02)
    C = sm_count()
    y = run(dep, plan, x, W, N, tc_tactic(dep, NT, C, 3, tile_k))
    T, KT = -(-N // 128), -(-K // tile_k)
    U = T * KT
    C = min(C, U)
    words = dep.dep_projection_plan_exchange(plan, C * 2 * NT * 128)
    assert words.size == C * 2 * NT * 128
    assert not (words >> np.uint64(32)).any()  # flags cleared for the next launch
    ws = (words & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.float32)
    checked = 0
    for t in range(T):
        segs = _stream_k_segments(U, C, KT, t)
        if len(segs) < 2:
            continue  # a whole tile: written straight from its accumulator
        rows = np.arange(128)
        n = t * 128 + rows
        keep = n < N
        for b in range(B):
            s = None
            for c, slot in segs:
                p = ws[((c * 2 + slot) * NT + b) * 128 + rows].astype(np.float32)
                s = p if s is None else (s + p).astype(np.float32)
            want = synth.bf16_from_f64(s.astype(np.float64))  # float32 -> float64 is exact
            np.testing.assert_array_equal(y[b, n[keep]], want[keep])
            checked += int(keep.sum())
    assert checked > 0


# ---------------- tensor-core tactic with fixed K pieces, dynamic items ----------------

def tcs_tactic(dep, NT, ctas, splits, stages=3, tile_k=128, max_rows=None, tile_n=128):
    return dep.dep_tactic_t(max_rows=max_rows or NT, kind=dep.DEP_KIND_TC_SPLIT, ctas=ctas, tile_n=tile_n,
                            tile_k=tile_k, stages=stages, cols=NT, splits=splits)


def tcs_plan(dep, N, K, tactics):
    """A plan whose workspace is grown for the given K-piece tactics."""
    plan = dep.dep_projection_plan(N, K, [1])
    for t in tactics:
        dep.dep_projection_plan_set(plan, t)
    return plan


TCS_STAGES = {(16, 64): 4, (16, 128): 3, (16, 256): 2, (32, 64): 4, (32, 256): 2, (64, 64): 4,
              (64, 128): 3, (128, 64): 4, (128, 128): 2, (256, 64): 3}


@pytest.mark.parametrize("N,K", [(128, 64), (333, 1000), (97, 264), (1000, 3000)])
@pytest.mark.parametrize("NT,tile_k", sorted(TCS_STAGES))
@pytest.mark.parametrize("BM", [128, 64])
def test_tcs_parity_vs_oracle(dep, orc, N, K, NT, tile_k, BM):
    """K-piece tensor-core kernel, every MMA width and stage width, MMA M of 128
    and 64 weight rows: one piece (direct stores), three pieces, and more pieces
    than k-tiles (capped); grids of one block, seven blocks and every SM (items
    taken dynamically); partial and full batches; ragged N and K tails."""
    st = TCS_STAGES[(NT, tile_k)]
    cases = [(1, 1), (1, sm_count()), (3, 1), (3, 7), (3, sm_count()), (64, sm_count())]
    plan = tcs_plan(dep, N, K, [tcs_tactic(dep, NT, c, s, st, tile_k, max_rows=300 + i, tile_n=BM)
                                for i, (s, c) in enumerate(cases)])
    try:
        W = synth.normal_bf16(N + NT + 7, 1, (N, K), sigma=0.02)
        for B in sorted({1, min(NT, 5), NT}):
            x = synth.normal_bf16(B + NT + 7, 2, (B, K))
            ref = orc.linear(x, W)
            for splits, ctas in cases:
                y = run(dep, plan, x, W, N, tcs_tactic(dep, NT, ctas, splits, st, tile_k, tile_n=BM))
                ok, worst, idx = within_tolerance(y, ref)
                assert ok, (B, splits, ctas, worst, idx)
        assert dep.dep_projection_device_status(plan) == 0
    finally:
        dep.dep_projection_plan_destroy(plan)


@pytest.mark.parametrize("NT,B,splits,BM", [(16, 16, 5, 128), (16, 3, 1, 128), (64, 40, 4, 128),
                                            (256, 256, 2, 128), (16, 16, 3, 64), (128, 77, 1, 64)])
def test_tcs_schedule_independent(dep, NT, B, splits, BM):
    """Which block runs which (tile, piece) item does not enter the arithmetic:
    grids of 1, 7, 40 and all SMs give identical bits, run after run and in a
    CUDA-graph replay."""
    N, K = 1000, 4096
    grids = [1, 7, 40, sm_count()]
    plan = tcs_plan(dep, N, K, [tcs_tactic(dep, NT, g, splits, 2, 128, max_rows=300 + i, tile_n=BM)
                                for i, g in enumerate(grids)])
    try:
        x = to_dev(synth.normal_bf16(60 + B, 2, (B, K)))
        W = to_dev(synth.normal_bf16(61, 1, (N, K), sigma=0.02))
        outs = []
        for g in grids:
            for _ in range(2):
                y = empty_out(B, N)
                dep.dep_projection_run_tactic(plan, tcs_tactic(dep, NT, g, splits, 2, 128, tile_n=BM), x, W, y, B)
                outs.append(y)
        ys = [empty_out(B, N) for _ in range(3)]
        tac = tcs_tactic(dep, NT, sm_count(), splits, 2, 128, tile_n=BM)
        torch.cuda.synchronize()  # a plan serves one stream at a time
        graph = torch.cuda.CUDAGraph()
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            dep.dep_projection_run_tactic(plan, tac, x, W, ys[0], B, stream)  # warm-up outside capture
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            for y in ys:
                dep.dep_projection_run_tactic(plan, tac, x, W, y, B, stream)
        graph.replay()
        graph.replay()
        torch.cuda.synchronize()
        outs += ys
        for y in outs[1:]:
            assert torch.equal(y.view(torch.int16), outs[0].view(torch.int16))
        assert dep.dep_projection_device_status(plan) == 0
    finally:
        dep.dep_projection_plan_destroy(plan)


@pytest.mark.parametrize("NT,B,tile_k", [(16, 8, 256), (32, 32, 64), (128, 100, 128)])
def test_tcs_one_piece_equals_whole_tile_stream_k(dep, NT, B, tile_k):
    """With one piece per tile each tile is summed by one accumulator over all of
    K in the same MMA sequence as the stream-K kernel launched with one block per
    tile: the two kernels give identical bits."""
    N, K = 1000, 3000
    T = -(-N // 128)
    plan = tcs_plan(dep, N, K, [tcs_tactic(dep, NT, sm_count(), 1, 2, tile_k, max_rows=300),
                                tc_tactic(dep, NT, T, 2, tile_k)])
    try:
        x = synth.normal_bf16(70 + B, 2, (B, K))
        W = synth.normal_bf16(71, 1, (N, K), sigma=0.02)
        y1 = run(dep, plan, x, W, N, tcs_tactic(dep, NT, sm_count(), 1, 2, tile_k))
        y2 = run(dep, plan, x, W, N, tc_tactic(dep, NT, T, 2, tile_k))
        np.testing.assert_array_equal(y1, y2)
    finally:
        dep.dep_projection_plan_destroy(plan)


@pytest.mark.parametrize("NT,B,splits,tile_k,BM", [(16, 16, 8, 256, 128), (16, 5, 3, 64, 128),
                                                   (64, 64, 4, 128, 128), (256, 200, 2, 64, 128),
                                                   (16, 16, 4, 256, 64), (32, 20, 3, 128, 64)])
def test_tcs_fixup_bitexact_from_partials(dep, NT, B, splits, tile_k, BM):
    """The K pieces' FP32 partials left in the exchange words, added in piece
    order 0..S-1 in float32 and rounded to BF16 (nearest, ties to even), give y
    bit for bit; every "full" flag is clear once the launch has finished."""
    N, K = 1000, 4096
    plan = tcs_plan(dep, N, K, [tcs_tactic(dep, NT, sm_count(), splits, 2, tile_k, tile_n=BM)])
    try:
        x = synth.normal_bf16(80 + NT, 2, (B, K))
        W = synth.normal_bf16(81, 1, (N, K), sigma=0.02)
        y = run(dep, plan, x, W, N, tcs_tactic(dep, NT, sm_count(), splits, 2, tile_k, tile_n=BM))
        T = -(-N // BM)
        S = min(splits, -(-K // tile_k))
        words = dep.dep_projection_plan_exchange(plan, T * S * NT * BM).reshape(T, S, NT, BM)
        assert not (words[:, :, :B, :] >> np.uint64(32)).any()  # flags cleared for the next launch
        ws = (words & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.float32)
        rows = np.arange(BM)
        for t in range(T):
            n = t * BM + rows
            keep = n < N
            s = ws[t, 0, :B, :].copy()
            for p in range(1, S):
                s = (s + ws[t, p, :B, :]).astype(np.float32)
            want = synth.bf16_from_f64(s.astype(np.float64))
            np.testing.assert_array_equal(y[:, n[keep]], want[:, keep])
    finally:
        dep.dep_projection_plan_destroy(plan)


@pytest.mark.parametrize("B,NT,splits,BM", [(40, 16, 2, 128), (300, 256, 1, 128), (33, 32, 3, 64)])
def test_tcs_batches_wider_than_the_mma(dep, orc, B, NT, splits, BM):
    """A batch wider than the MMA's N runs as consecutive launches of NT rows of x
    each (the last one ragged), every launch reusing the plan's item counter and
    piece counters: all rows match the oracle and a second run gives the same bits."""
    N, K = 700, 2048
    t = tcs_tactic(dep, NT, sm_count(), splits, 2, 128, max_rows=B, tile_n=BM)
    plan = tcs_plan(dep, N, K, [t])
    try:
        x = synth.normal_bf16(100 + B, 2, (B, K))
        W = synth.normal_bf16(101, 1, (N, K), sigma=0.02)
        y1 = run(dep, plan, x, W, N)
        y2 = run(dep, plan, x, W, N)
        np.testing.assert_array_equal(y1, y2)
        ok, worst, idx = within_tolerance(y1, orc.linear(x, W))
        assert ok, (worst, idx)
        assert dep.dep_projection_plan_query(plan, B).kind == dep.DEP_KIND_TC_SPLIT
        assert dep.dep_projection_device_status(plan) == 0
    finally:
        dep.dep_projection_plan_destroy(plan)


def test_exchange_give_up_is_reported_and_cleared(dep, orc):
    """The split-K exchange's bounded wait, made to run out without faulting
    anything: the self-test leaves published exchange words and a counter
    behind and has the reducer wait for a piece nobody publishes.  The give-up
    comes back as DEP_DEV_TIMEOUT_EPILOGUE; reading the status clears the
    exchange region and the counters; afterwards the K-piece tensor-core
    kernel, the split-K FMA kernel and the wide-batch stream-K kernel give the
    bits of a fresh plan (a stale flag or counter would change them)."""
    N, K, B = 7168, 4096, 16
    x = synth.normal_bf16(51, 2, (B, K))
    W = synth.normal_bf16(52, 1, (N, K), sigma=0.02)
    sms = sm_count()
    fma = fma_tactic(dep, 8, sms)
    wide = dep.dep_tactic_t(max_rows=64, kind=dep.DEP_KIND_TC_WIDE, ctas=sms, tile_n=256, tile_k=64, stages=4,
                            cols=64)
    pieces = tcs_tactic(dep, 16, sms, 2, 3, 256, max_rows=B)  # 128-row tiles in two K pieces: exchanged

    def all_runs(plan):
        return [run(dep, plan, x, W, N), run(dep, plan, x, W, N, fma), run(dep, plan, x, W, N, wide)]

    fresh = dep.dep_projection_plan(N, K, [B])
    plan = dep.dep_projection_plan(N, K, [B])
    try:
        for p_ in (fresh, plan):
            dep.dep_projection_plan_set(p_, wide)
            dep.dep_projection_plan_set(p_, pieces)
        assert dep.dep_projection_plan_query(plan, B).kind == dep.DEP_KIND_TC_SPLIT
        want = all_runs(fresh)
        assert dep.dep_projection_device_status(fresh) == 0
        ok, worst, idx = within_tolerance(want[0], orc.linear(x, W))
        assert ok, (worst, idx)
        dep.dep_projection_plan_selftest_exchange(plan, 2000)  # 2 ms limit
        assert dep.dep_projection_device_status(plan) == dep.DEP_DEV_TIMEOUT_EPILOGUE
        words = dep.dep_projection_plan_exchange(plan, 4 * 16 * 32)
        assert not words.any()  # flags and values cleared
        for got, ref in zip(all_runs(plan), want):
            np.testing.assert_array_equal(got, ref)
        assert dep.dep_projection_device_status(plan) == 0
    finally:
        dep.dep_projection_plan_destroy(plan)
        dep.dep_projection_plan_destroy(fresh)


@pytest.mark.parametrize("kind,NT,tile_n,tile_k,B", [("split", 16, 128, 256, 16), ("split", 16, 64, 256, 5),
                                                     ("split", 32, 64, 128, 20), ("gemm", 16, 128, 128, 9),
                                                     ("gemm", 64, 128, 128, 64)])
def test_stage_copy_forms_agree_bitwise(dep, kind, NT, tile_n, tile_k, B):
    """A K that is a multiple of 64 loads each stage with one copy of a column-block
    view of W and x; any other K loads it slice by slice through 2-D maps that
    zero-fill past column K.  The same product with 8 zero columns appended to x
    and W (K = 4104) takes the second form and only adds zero products to each
    accumulator, so with one piece per tile the two give identical bits."""
    N, K, pad = 1000, 4096, 8
    x = synth.normal_bf16(90 + NT, 2, (B, K))
    W = synth.normal_bf16(91, 1, (N, K), sigma=0.02)
    xp = np.concatenate([x, np.zeros((B, pad), np.uint16)], axis=1)
    Wp = np.concatenate([W, np.zeros((N, pad), np.uint16)], axis=1)
    tiles = -(-N // tile_n)
    if kind == "split":
        t = tcs_tactic(dep, NT, sm_count(), 1, 2, tile_k, max_rows=B, tile_n=tile_n)
    else:
        t = tc_tactic(dep, NT, tiles, 2, tile_k)
        t.max_rows = B
    got = []
    for k_, xx, ww in ((K, x, W), (K + pad, xp, Wp)):
        plan = tcs_plan(dep, N, k_, [t])
        try:
            got.append(run(dep, plan, xx, ww, N, t))
            assert dep.dep_projection_device_status(plan) == 0
        finally:
            dep.dep_projection_plan_destroy(plan)
    np.testing.assert_array_equal(got[0], got[1])


def test_grid_larger_than_the_device_holds_is_refused(dep):
    """Kinds whose blocks wait on one another need the whole grid resident: a
    tactic asking for more blocks than the device holds at once is refused by
    plan_set and run_tactic, and the plan keeps its table."""
    N, K = 7168, 4096
    plan = dep.dep_projection_plan(N, K, [16])
    try:
        before = dep.dep_projection_plan_query(plan, 16).as_dict()
        too_many = tc_tactic(dep, 16, 8 * sm_count(), 4, 64)  # 448 tiles x 64 units: enough units
        too_many.max_rows = 16
        with pytest.raises(dep.DepError) as e:
            dep.dep_projection_plan_set(plan, too_many)
        assert e.value.status == dep.DEP_ERR_UNSUPPORTED
        assert dep.dep_projection_plan_query(plan, 16).as_dict() == before
        x, W = synth.normal_bf16(1, 2, (16, K)), synth.normal_bf16(2, 1, (N, K), sigma=0.02)
        with pytest.raises(dep.DepError) as e:
            run(dep, plan, x, W, N, too_many)
        assert e.value.status == dep.DEP_ERR_UNSUPPORTED
    finally:
        dep.dep_projection_plan_destroy(plan)
