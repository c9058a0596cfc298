"""The C++ example (include/msa_example.cu) runs the three entry points through
the C ABI alone, with library-sized workspaces, and checks every status and
that the whole output was written."""
import subprocess

import pytest

from tests.test_abi import _build_c_example

pytestmark = pytest.mark.gpu


def test_c_example_runs(tmp_path):
    exe = tmp_path / "msa_example"
    r = _build_c_example(exe)
    assert r.returncode == 0, r.stderr[-2000:]
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "msa_example ok" in run.stdout
