"""Runs of every tactic kind on ragged shapes through the bounds-checked
(DEP_DEBUG) library; executed in a child process by test_gpu_debug_build.py
(the binding loads one library per process).  Prints one line per run and
exits nonzero on the first failure."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import skinny_bf16_split_gb300._binding as binding  # noqa: E402
from skinny_bf16_split_gb300 import build  # noqa: E402

binding.LIB_PATH = build.build(debug=True)
import skinny_bf16_split_gb300 as dep  # noqa: E402
import oracle  # noqa: E402
from gpu_util import empty_out, to_dev, to_host  # noqa: E402
from helpers import within_tolerance  # noqa: E402
from skinny_bf16_split_gb300 import synth  # noqa: E402


def main():
    torch.cuda.set_device(0)
    assert os.path.samefile(dep.lib()._name, binding.LIB_PATH)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    T = dep.dep_tactic_t

    def tactics(N):
        g2 = -(-N // 256)
        return [
            ("fma", T(max_rows=4, kind=dep.DEP_KIND_SPLITK_FMA, ctas=7, tile_n=32, tile_k=256, stages=4, cols=4)),
            ("fma-all", T(max_rows=8, kind=dep.DEP_KIND_SPLITK_FMA, ctas=sms, tile_n=32, tile_k=256, stages=6,
                          cols=8)),
            ("rows", T(max_rows=2, kind=dep.DEP_KIND_ROWS, ctas=sms, tile_n=16, tile_k=1024, stages=2, cols=2)),
            ("tc", T(max_rows=32, kind=dep.DEP_KIND_TC, ctas=7, tile_n=128, tile_k=128, stages=3, cols=32)),
            ("tc-all", T(max_rows=64, kind=dep.DEP_KIND_TC, ctas=sms, tile_n=128, tile_k=64, stages=4, cols=64)),
            ("k-pieces", T(max_rows=16, kind=dep.DEP_KIND_TC_SPLIT, ctas=sms, tile_n=128, tile_k=128, stages=3,
                           cols=16, splits=3)),
            ("k-pieces-64", T(max_rows=16, kind=dep.DEP_KIND_TC_SPLIT, ctas=sms, tile_n=64, tile_k=64, stages=3,
                              cols=16, splits=5)),
            ("k-pieces-64-whole", T(max_rows=16, kind=dep.DEP_KIND_TC_SPLIT, ctas=sms, tile_n=64, tile_k=256,
                                    stages=5, cols=16, splits=1)),
            ("k-pieces-5", T(max_rows=16, kind=dep.DEP_KIND_TC_SPLIT, ctas=sms, tile_n=128, tile_k=256, stages=3,
                             cols=16, splits=5)),
            ("wide", T(max_rows=64, kind=dep.DEP_KIND_TC_WIDE, ctas=sms, tile_n=256, tile_k=64, stages=4, cols=64)),
            ("cluster-2", T(max_rows=128, kind=dep.DEP_KIND_TC_CLUSTER, ctas=2 * g2, tile_n=256, tile_k=64, stages=5,
                            cols=128, splits=2)),
            ("cluster-3", T(max_rows=256, kind=dep.DEP_KIND_TC_CLUSTER, ctas=3 * g2, tile_n=256, tile_k=64,
                            stages=4, cols=256, splits=3)),
            ("cluster-192", T(max_rows=512, kind=dep.DEP_KIND_TC_CLUSTER, ctas=2 * -(-N // 192), tile_n=192,
                              tile_k=64, stages=5, cols=256, splits=2)),
            ("x-on-m", T(max_rows=1024, kind=dep.DEP_KIND_TC_XM, ctas=7, tile_n=48, tile_k=128, stages=3,
                         cols=128)),
            ("x-on-m-2", T(max_rows=2048, kind=dep.DEP_KIND_TC_XM, ctas=sms, tile_n=96, tile_k=64, stages=3,
                           cols=256)),
            ("x-on-m-pairs", T(max_rows=4096, kind=dep.DEP_KIND_TC_XM, ctas=6, tile_n=64, tile_k=64, stages=4,
                               cols=256, splits=2)),
            ("warp-mma", T(max_rows=8192, kind=dep.DEP_KIND_WARP_MMA, ctas=1, tile_n=16, tile_k=256, stages=3,
                           cols=16)),
            ("warp-mma-pieces", T(max_rows=16384, kind=dep.DEP_KIND_WARP_MMA, ctas=1, tile_n=16, tile_k=128,
                                  stages=4, cols=16, splits=4)),
        ]

    # K = 2048 and 1088 (multiples of 64) take the one-copy column-block stage
    # loads, 1088 with a last 256-column stage past the end; the others the
    # per-slice 2-D loads.
    for N, K, B in [(333, 1000, 5), (97, 264, 33), (1000, 3000, 100), (1024, 2048, 255), (333, 1088, 16)]:
        x = synth.normal_bf16(N + B, 2, (B, K))
        W = synth.normal_bf16(N + K, 1, (N, K), sigma=0.02)
        ref = oracle.linear(x, W)
        plan = dep.dep_projection_plan(N, K, [1, 2, 8, 16, 32, 64, 128, 256])
        try:
            for name, t in tactics(N):
                dep.dep_projection_plan_set(plan, t)  # room for every tactic's workspace
            xd, Wd = to_dev(x), to_dev(W)
            runs = [("default", None)] + tactics(N)
            for name, t in runs:
                y = empty_out(B, N)
                if t is None:
                    dep.dep_projection_run(plan, xd, Wd, y, B)
                else:
                    dep.dep_projection_run_tactic(plan, t, xd, Wd, y, B)
                torch.cuda.synchronize()
                code = dep.dep_projection_device_status(plan)
                ok, worst, idx = within_tolerance(to_host(y), ref)
                print(f"N={N} K={K} B={B} {name}: status {code}, within tolerance {ok}", flush=True)
                if code != 0 or not ok:
                    return 1
        finally:
            dep.dep_projection_plan_destroy(plan)
    return 0


if __name__ == "__main__":
    sys.exit(main())
