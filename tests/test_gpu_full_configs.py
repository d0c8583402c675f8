"""Parity at the workloads' full sizes, in the launch configuration bench.py times.

Workloads (skinny_bf16_split_gb300.synth): the DSA packed input projection at
B = 1 (unit-RMS rows), the o_proj sweep, the KDA packed input projection sweep,
the wide-batch DSA projection, the 8-layer decode chain -- the weights the
runtime.dep page lists (DSA 14560 x 7168, o_proj 7168 x 12288, KDA 49376 x 7168)
-- plus verify-step batches B = requests x q (runtime.dep page, DepKda: verify
keys (B // q, q)) and TP-G shards of the same weights (runtime.hybrid page,
HybridAttention.__init__: projection_policies(tp, pitch, ...), o_proj 12288 // tp).

Each call runs through the default plan for its shape and batch set (as the
benchmark does) and is checked against the exact oracle on sampled weight rows:
every tile boundary of both kernels' tile sizes, the first and last rows, and
random rows.  The tolerance's rms is taken over the sampled reference outputs.
Every full output is also checked for properties that hold at any size: it is
written everywhere (no NaN left from the pre-filled buffer), a second run gives
the same bits, and its spread matches 0.02 sqrt(K) for N(0,1) x N(0,0.02) inputs.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gpu_util import empty_out, to_dev, to_host  # noqa: E402
from helpers import within_tolerance  # noqa: E402
from skinny_bf16_split_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu


def sample_rows(N, seed):
    rng = np.random.default_rng(seed)
    edges = set()
    for tn in (32, 64, 128):
        for t in range(0, N, tn):
            edges.update((t, min(N - 1, t + tn - 1)))
    edges = sorted(edges)
    if len(edges) > 1200:  # keep the oracle's work bounded: a spread of boundaries
        edges = [edges[i] for i in np.linspace(0, len(edges) - 1, 1200).astype(int)]
    rand = rng.choice(N, min(N, 400), replace=False)
    return np.unique(np.concatenate([edges, rand, [0, N - 1]])).astype(np.int64)


@pytest.fixture(scope="module")
def weights():
    cache = {}

    def get(call):
        if call.weight_key not in cache:
            cache.clear()  # one full-size weight on the host at a time
            cache[call.weight_key] = call.weight()
        return cache[call.weight_key]
    return get


@pytest.mark.parametrize("workload", [w for w in synth.WORKLOADS if w != "baseline"])  # its parts, one by one
def test_workload_full_size(dep, orc, weights, workload):
    calls = synth.workload(workload)
    batches = {}
    for c in calls:
        batches.setdefault((c.N, c.K), set()).add(c.B)
    from bench import TUNED_BY_DEFAULT  # the launch configuration the bench times: tuned where it
    # tunes, programmatic dependent launch, calls back to back on one stream
    flags = (dep.DEP_PLAN_TUNE if workload in TUNED_BY_DEFAULT else dep.DEP_PLAN_DEFAULT) | dep.DEP_PLAN_PDL
    plans = {k: dep.dep_projection_plan(k[0], k[1], sorted(v), flags) for k, v in batches.items()}
    try:
        for i, c in enumerate(calls):
            W = weights(c)
            x = c.activations()
            Wd, xd = to_dev(W), to_dev(x)
            plan = plans[(c.N, c.K)]
            y1 = empty_out(c.B, c.N)
            dep.dep_projection_run(plan, xd, Wd, y1, c.B)
            y2 = empty_out(c.B, c.N)
            dep.dep_projection_run(plan, xd, Wd, y2, c.B)
            torch.cuda.synchronize()
            got = to_host(y1)
            assert torch.equal(y1.view(torch.int16), y2.view(torch.int16)), c.name
            f = synth.bf16_to_f32(got)
            assert not np.isnan(f).any(), c.name
            sd = float(f.std())
            assert abs(sd / (0.02 * np.sqrt(c.K)) - 1) < 0.1, (c.name, sd)
            rows = sample_rows(c.N, i)
            ref = orc.linear_rows(x, W, rows)
            ok, worst, idx = within_tolerance(got[:, rows], ref)
            assert ok, (c.name, worst, idx)
            del Wd, xd, y1, y2
        for p in plans.values():
            assert dep.dep_projection_device_status(p) == 0
    finally:
        for p in plans.values():
            dep.dep_projection_plan_destroy(p)


@pytest.mark.slow
def test_dsa_b1_every_output_against_the_oracle(dep, orc):
    """DSA packed input projection at B = 1 (x with unit-RMS rows), the benchmark's
    first configuration at full size: all 14,560 outputs of the default plan's
    call against the exact oracle's, element by element (about half a minute of
    oracle work on the host's cores), and run to run bit for bit."""
    c = synth.workload("dsa_b1")[0]
    W, x = c.weight(), c.activations()
    plan = dep.dep_projection_plan(c.N, c.K, [1])
    try:
        Wd, xd = to_dev(W), to_dev(x)
        y1, y2 = empty_out(1, c.N), empty_out(1, c.N)
        dep.dep_projection_run(plan, xd, Wd, y1, 1)
        dep.dep_projection_run(plan, xd, Wd, y2, 1)
        torch.cuda.synchronize()
        assert dep.dep_projection_device_status(plan) == 0
    finally:
        dep.dep_projection_plan_destroy(plan)
    got = to_host(y1)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    ref = orc.linear(x, W)
    ok, worst, idx = within_tolerance(got, ref)
    assert ok, (worst, idx)
    # the default tactic at one row is the whole-row kernel, whose order the FP32 mirror restates
    np.testing.assert_array_equal(got, orc.mirror_fma(x, W, 1, 64))
