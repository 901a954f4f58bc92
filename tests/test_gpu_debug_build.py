"""The debug build, libringattn_debug.so: the same kernels, with every raw global
load and store of the ring, step, backward and decode kernels checking its index
range first (a failed check records RA_ERR_BOUNDS and skips the access). The
small-case GPU parity suites run again on it in a child process with RA_DEBUG=1:
they assert a clean status word after every call, so any failed check fails them,
and their results must still match the oracle."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ra = pytest.importorskip("online_softmax_merge_gb300")
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
IN_DEBUG = os.environ.get("RA_DEBUG") == "1"


def test_selftest_bounds_fires_only_in_the_debug_build():
    assert ra.debug_checks() == IN_DEBUG
    ra.selftest_bounds(DEV)
    torch.cuda.synchronize(DEV)
    assert ra.last_error(DEV) == (ra.RA_ERR_BOUNDS if IN_DEBUG else 0)
    assert ra.last_error(DEV) == 0                  # reading cleared it


@pytest.mark.skipif(IN_DEBUG, reason="this process already runs the debug build")
def test_small_case_gpu_suites_pass_on_the_debug_build():
    files = ["tests/test_gpu_parity.py", "tests/test_gpu_step_merge.py",
             "tests/test_gpu_decode.py", "tests/test_gpu_bwd.py", "tests/test_gpu_fuzz.py",
             "tests/test_gpu_maps.py", "tests/test_gpu_debug_build.py"]
    env = dict(os.environ, RA_DEBUG="1")
    r = subprocess.run([sys.executable, "-m", "pytest", *files, "-m", "gpu", "-q", "-x",
                        "-p", "no:cacheprovider", "-k", "not sampled and not 128k"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
