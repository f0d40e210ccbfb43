"""The checked build (libgemm_gather_checked.so: the gather kernels with
device-side bounds and table checks, GG_CHECKED=1) on a GB300, in a child
process that loads it (GEMM_GATHER_CHECKED=1 at import):

* every whole-heap parity test of the all-gather and of the neighbouring
  collectives passes under it with the status words clear (the checks never
  fire on valid arguments and change no result);
* the planted wrong table entries of test_gpu_checked_table.py are reported
  as GG_ERR_NOT_IN_HEAP and not used."""
import os
import re
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _child(files, timeout):
    env = dict(os.environ, GEMM_GATHER_CHECKED="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "tests.checked_plugin",
           "-p", "no:cacheprovider", *files]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)
    tail = (r.stdout + r.stderr)[-4000:]
    assert r.returncode == 0, tail
    m = re.search(r"(\d+) passed", r.stdout)
    assert m, tail
    return int(m.group(1)), tail


def test_parity_suites_pass_under_the_checked_build():
    passed, tail = _child(["tests/test_gpu_all_gather.py", "tests/test_gpu_collectives.py",
                           "tests/test_gpu_balance.py"], timeout=1500)
    assert passed >= 100, tail


def test_planted_table_faults_are_reported():
    passed, tail = _child(["tests/test_gpu_checked_table.py"], timeout=600)
    assert passed == 7 * 3 + 2, tail
    assert "skipped" not in tail.splitlines()[-1], tail
