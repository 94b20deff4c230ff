"""The profile build (libmoe_profile.so, compiled with -DMOE_PROFILE by
__graft_entry__.build()): its outputs are bit-exact with the oracle and its
kernels fill the phase slots. It runs in a child process, which loads the
profile library in place of the default one."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_profile_build_outputs_and_slots():
    from combine_moe_layout_02_gb300 import build as moe_build

    moe_build.build(variant="profile")
    env = dict(os.environ, MOE_LIBRARY="profile")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "profile_run.py")], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-3000:]
    assert "profile ok" in r.stdout
