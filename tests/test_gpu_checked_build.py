"""The GPU parity suite once more against the bounds-checked build of the library.

``libtwell_check.so`` is the same library compiled with -DTW_CHECK: every index a
kernel computes from data it reads (neuron indices of the formats, token rows of the
row gathers and scatters, slots of the transposed Hybrid's records, counts that size
a loop) is compared with the size of the buffer it addresses; a violation raises
TW_EBOUNDS in the status word, prints its source line and skips the access instead
of touching memory. The suite runs in a child process that loads the checked build
(TW_LIB_PATH); it must pass, and no violation may be printed."""
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_gpu_suite_under_the_bounds_checked_build():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    sys.path.insert(0, ROOT)
    from activation_sparse_feedforward_gb300.build import build

    path = build(check=True)
    env = dict(os.environ, TW_LIB_PATH=path)
    here = os.path.basename(__file__)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests"), "-m", "gpu", "-x", "-q", "-s",
                        "-p", "no:cacheprovider", "--deselect", f"tests/{here}::test_gpu_suite_under_the_bounds_checked_build"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    out = r.stdout + r.stderr
    assert "TW_CHECK: index out of bounds" not in out, out[-4000:]
    assert r.returncode == 0, out[-4000:]
    assert " passed" in out
