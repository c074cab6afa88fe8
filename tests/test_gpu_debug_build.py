"""The debug build (ADACOMP_DEBUG_CHECKS=1: libadacomp_debug.so, every call waits for its
stream and reports its kernels' errors) runs the smoke case, compress of three learners
and their decode, bit for bit as the oracle does."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_debug_build_matches_the_oracle():
    code = ("import __graft_entry__ as g, residual_gradient_compression_gb300 as ac, os; g.smoke(); "
            "print('lib', os.path.basename(ac._LIB_PATH))")
    env = dict(os.environ, ADACOMP_DEBUG_CHECKS="1")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "smoke ok" in r.stdout and "lib libadacomp_debug.so" in r.stdout, r.stdout
