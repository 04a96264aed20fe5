"""The debug build of the library (compiled with FOS_DEBUG): its kernels check the stage
offsets, tensor-memory columns and row indices they are about to use, and a check that fails
records FOS_ERR_INDEX in the device error word and skips the access, instead of trapping.  It
stands in for a memory checker on the GPU: the small parity grid, the one-warp-per-row and
row-group kernels and the fused sink gradient run on it in a child process (FOS_LIBRARY=debug
selects the library), and every one of those tests ends by asserting that the device error word
is clear."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def run_child(args, timeout=1500):
    env = dict(os.environ, FOS_LIBRARY="debug")
    return subprocess.run([sys.executable, *args], env=env, cwd=ROOT, capture_output=True,
                          text=True, timeout=timeout)


def test_suites_pass_on_the_debug_build():
    from deterministic_attention_softmax_gb300 import _build

    _build.build(debug=True)
    # the child really runs the debug library
    probe = run_child(["-c", "import deterministic_attention_softmax_gb300._abi as a; "
                             "print(a.LIB_PATH); a.lib()"])
    assert probe.returncode == 0 and probe.stdout.strip().endswith("libfos_softmax_debug.so"), \
        probe.stdout + probe.stderr
    tests = [os.path.join(HERE, f) for f in ("test_parity_small.py", "test_rowwarp.py",
                                             "test_bwd_sink.py")]
    tests.append(os.path.join(HERE, "test_invariance.py") +
                 "::test_row_groups_per_cta_give_the_same_bits")
    r = run_child(["-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider", *tests])
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
