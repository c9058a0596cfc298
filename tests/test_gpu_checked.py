"""The bounds-checking build (libmsa_checked.so, compiled with MSA_CHECKED).

Every index the kernels read from index data (tile distances, chunk and
column positions, kept-block ids, item lists and their counts) is checked
against its buffer there; a bad one is replaced by a valid index and reported
as MSA_ERR_BOUNDS in the device status word, with no trap.  This test runs the
small GPU parity suites against that build, with every call's device status
read back (MSA_STRICT_STATUS): the parity must hold and no check may fire.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SUITES = ["tests/test_gpu_parity.py", "tests/test_gpu_edge_cases.py", "tests/test_gpu_hip.py",
          "tests/test_gpu_ragged.py", "tests/test_gpu_kv.py", "tests/test_gpu_layouts.py"]


@pytest.mark.gpu
def test_parity_suites_under_the_bounds_checking_build():
    from dynamic_sparse_attention_slash_gb300 import build
    lib = build.build(checked=True)
    env = dict(os.environ, MSA_LIBRARY=lib, MSA_STRICT_STATUS="1")
    probe = subprocess.run(
        [sys.executable, "-c", "from dynamic_sparse_attention_slash_gb300 import msa; "
         "msa.load_library(); print(msa.LIB_PATH, msa.STRICT_STATUS)"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert probe.stdout.split() == [lib, "True"], probe.stdout + probe.stderr
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "-m", "gpu", "-k", "not two_slabs and not full_size", *SUITES],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and " failed" not in r.stdout
