"""The debug build (libmoe_debug.so: every index a kernel takes from the
dispatch checked against its bounds, a failed check recorded in the error
word instead of trapping) runs clean on layers that cover every kernel
family, each checked against the oracle.  It runs in a child process, which
loads the debug library in place of libmoe.so."""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.mark.gpu
def test_debug_build_runs_clean_against_the_oracle():
    sys.path.insert(0, ROOT)
    from expert_routed_ffn_gemm_gb300 import build

    build.build(variants=("debug",))
    env = dict(os.environ, MOE_LIBRARY="debug")
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_cases.py")], env=env, capture_output=True,
                       text=True, timeout=900)
    print(r.stdout)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert r.stdout.count("ok  ") == 10
