"""The bounds-checked build (DEP_DEBUG): every kernel checks each index into y,
the plan's workspace and shared memory before it uses it, and records
DEP_DEV_BOUNDS (skipping the access) instead of touching memory it does not
own.  This test builds that variant and runs every tactic kind on ragged
shapes through it (in a child process: the binding loads one library per
process); every run must match the oracle and leave the status word at 0."""
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_every_kind_on_ragged_shapes_under_bounds_checks():
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_build_runs.py")], capture_output=True,
                       text=True, timeout=1200)
    print(r.stdout[-4000:])
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert r.stdout.count("status 0, within tolerance True") == 5 * 19  # 5 shapes x (default + 18 tactics)
