"""GPU: the tensor-memory (tcgen05) history kernel on pools of group size 128.  Those pools normally run the
warp-MMA kernel; OSCAR_DECODE_TC=1 routes them to the tensor-memory kernel (its one-group form, G = 4 and 8
query heads per KV head), and the whole decode parity suite then runs against the oracle on it, in a child
process whose environment sets the variable (the library reads it once per process)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_decode_suite_on_the_tensor_memory_kernel():
    env = dict(os.environ, OSCAR_DECODE_TC="1")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join("tests", "test_gpu_decode.py"), "-q", "-x",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
