"""The index-checked build of the library on the GPU: in a child process that
loads it (W4A16_LIBRARY=checked), every kernel family runs on parity cases
(ragged shapes, a K split, a two-layer sequence with and without SwiGLU,
attention, W4A8) within the oracle's tolerance, and no index check fails
(W4A16_DEV_INDEX stays clear).  This stands in for a memory checker: every
checked access skips itself and sets a status bit instead of faulting."""
import json
import os
import subprocess
import sys

import pytest

from int4_weight_only_gemv_gb300 import build as wbuild

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_checked_build_runs_clean():
    wbuild.build()
    path = wbuild.build(checked=True)
    env = dict(os.environ, W4A16_LIBRARY="checked")
    r = subprocess.run([sys.executable, os.path.join(HERE, "gpu_checked_run.py")], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    rep = json.loads(r.stdout.strip().splitlines()[-1])
    assert rep["lib"] == path
    assert rep["fail"] == [], rep
    assert rep["status"] == 0, rep
