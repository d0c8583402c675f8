"""The no-allocation entry point, dep_projection_run_static, against the mirror, oracle and plan path.

Callers that must not allocate device memory -- code inside a device-memory
allocator or pool, hosts that reserve all device memory up front, paths that
cannot take cudaMalloc's implicit synchronisation -- cannot build a plan, since
a plan allocates its workspace.  dep_projection_run_static serves them with a
fixed scratch array compiled into the library.  This test calls it through the
C ABI three times in a row, on different problems, and checks each output bit
for bit against the FP32 mirror of the kernel it runs, and within the acceptance
tolerance of the tests against the exact oracle and the plan-based
dep_projection_run.

The file is named so that pytest collects it last: if it fails, a run that stops
at the first failure has already run every other test.  It also passes alone in
a fresh process (the library and the CUDA context are set up by fixtures).
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


def test_static_scratch_entry_matches_plan_entry(dep, orc):
    """Three calls in a row on one stream, then three checks per output: bit for
    bit against the FP32 mirror of the split-K FMA kernel the entry runs (32-row
    tiles, 256-column k-tiles, one block per SM), within the acceptance
    tolerance of the exact oracle, and within it of the plan-based
    dep_projection_run.  The 13-row batch runs as two passes of 8 rows, so its
    second pass reuses the tile counters and partials the first pass left."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    problems = [(3, 1000, 3000, 11), (8, 7168, 4096, 12), (13, 777, 2000, 13)]  # (B, N, K, seed)
    outs = []
    for B, N, K, seed in problems:
        xh = synth.normal_bf16(seed, synth.X_ID, (B, K))
        Wh = synth.normal_bf16(seed, synth.W_ID, (N, K), sigma=0.02)
        x, W = to_dev(xh), to_dev(Wh)
        y = empty_out(B, N)
        dep.dep_projection_run_static(x, W, y, N, K, B)
        outs.append((y, x, W, xh, Wh, B, N, K))
    torch.cuda.synchronize()
    for y, x, W, xh, Wh, B, N, K in outs:
        got = to_host(y)
        units = -(-N // 32) * -(-K // 256)
        np.testing.assert_array_equal(got, orc.mirror_fma(xh, Wh, min(sms, units), 32))
        ok, worst, idx = within_tolerance(got, orc.linear(xh, Wh))
        assert ok, (B, N, K, worst, idx)
        plan = dep.dep_projection_plan(N, K, [B])
        try:
            ref = empty_out(B, N)
            dep.dep_projection_run(plan, x, W, ref, B)
            torch.cuda.synchronize()
        finally:
            dep.dep_projection_plan_destroy(plan)
        ok, worst, idx = within_tolerance(got, to_host(ref))
        assert ok, (B, N, K, worst, idx)


def test_static_scratch_entry_rejects_oversized_and_bad_arguments(dep):
    """Refusals come back as status codes.  Every buffer is real and sized for the
    call it is passed to, so nothing here could touch memory it does not own."""
    K = 64
    x = torch.zeros(2, K, dtype=torch.bfloat16, device="cuda")
    N_big = 300000  # more weight rows than the fixed scratch array serves (262144)
    W_big = torch.zeros(N_big, K, dtype=torch.bfloat16, device="cuda")
    y_big = torch.zeros(2, N_big, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dep.DepError) as e:
        dep.dep_projection_run_static(x, W_big, y_big, N_big, K, 2)
    assert e.value.status == dep.DEP_ERR_UNSUPPORTED
    del W_big, y_big
    W = torch.zeros(64, K, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(2, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dep.DepError) as e:  # K not a multiple of 8
        dep.dep_projection_run_static(x, W, y, 64, 60, 2)
    assert e.value.status == dep.DEP_ERR_MISALIGNED
    with pytest.raises(dep.DepError) as e:  # y overlapping x (same size, so in bounds anyway)
        dep.dep_projection_run_static(x, W, x, 64, K, 2)
    assert e.value.status == dep.DEP_ERR_INVALID_ARG
    dep.dep_projection_run_static(x, W, y, 64, K, 0)  # B == 0: nothing to do
    torch.cuda.synchronize()
