"""The bounds-checked build (libhicache_checked.so, HICACHE_CHECKED=1): every
transfer kernel checks each decoded vector against the device buffers, the
host pool and the run table before touching it, and records a failure in a
device word instead of the access.  The randomised corpora -- 300 transfer
cases, 150 buffer groups, 100 call sequences of every kind -- and the
tensor-parallel, pipelined, chained and large-call tests run against the
checked library in a child process (valid inputs only), and every test must leave the check words
at zero (tests/conftest.py); their oracle comparisons run as usual."""
import os
import subprocess
import sys

import pytest
import torch

from tiered_kv_cache_gb300 import build as hc_build

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CORPORA = ["tests/test_gpu_fuzz.py", "tests/test_gpu_group_fuzz.py", "tests/test_gpu_sequence.py",
           "tests/test_gpu_tp.py", "tests/test_gpu_pipelined.py", "tests/test_gpu_group.py",
           "tests/test_gpu_chained.py", "tests/test_gpu_large_calls.py", "tests/test_gpu_wait_fuzz.py"]


def test_corpora_under_the_bounds_checked_build():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    hc_build.build()
    env = dict(os.environ, HICACHE_CHECKED="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider"]
                       + CORPORA, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and " failed" not in r.stdout
