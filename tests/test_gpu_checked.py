"""The checked build (-DMOE_CHECKED): the kernels check every index they form
from routing, bucket and segment data before the access it guards and set
MOE_STATUS_OUT_OF_BOUNDS instead of touching memory outside their buffers. It
is built here and run in a child process (the binding loads one library per
process), through every rail on a tiny and a gpt-oss-shaped layer: no check may
fire on valid inputs and every result must meet its rail's bound."""

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_checked_build_runs_every_rail_clean():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_moe_build", os.path.join(ROOT, "mxfp4_mixture_experts_bucket_gb300", "build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    lib = b.build(checked=True)
    assert os.path.exists(lib)
    env = dict(os.environ, MOE_MXFP4_CHECKED="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "checked_child.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "checked build ok" in r.stdout
