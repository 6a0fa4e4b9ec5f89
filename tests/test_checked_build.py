"""The bounds-checked build (WC_CHECKED=1) on the GPU.

Every kernel of that build compares each global load and store with the
extent of its buffer and skips, and counts, any access that would fall
outside.  First the records themselves are shown to work (one deliberate
violation per kernel file, made without touching memory, reaches the host
and is cleared).  Then the parity suites run against the checked library in
a child process; after every test the count must be zero, and the results
must still match the oracle."""
import os
import re
import subprocess
import sys
from pathlib import Path

import pytest

from weight_communication_gb300 import build

pytestmark = pytest.mark.gpu

ROOT = Path(__file__).resolve().parent.parent
KERNEL_FILES = 5        # qgz_quant, qgz_reduce, qgz_hop1, qgz_fused, qwz

PROBE = """
import sys
from weight_communication_gb300 import binding
n = binding.checked_violations(reset=True, probe=True)
msg = binding.last_error()
after = binding.checked_violations()
print(n, after, msg)
sys.exit(0 if (n == {files} and after == 0 and ".cu line" in msg) else 1)
"""


@pytest.fixture(scope="module")
def checked_env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = build.build(checked=True)
    return dict(os.environ, WC_LIBRARY=str(lib), WC_EXPECT_CHECKED="1")


def test_violation_records_reach_the_host(checked_env):
    proc = subprocess.run([sys.executable, "-c", PROBE.format(files=KERNEL_FILES)], cwd=ROOT,
                          env=checked_env, capture_output=True, text=True, timeout=300)
    assert proc.returncode == 0, proc.stdout + proc.stderr


def test_parity_suites_stay_in_bounds(checked_env):
    proc = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu",
                           "-p", "no:cacheprovider", "tests/test_parity_qgz.py",
                           "tests/test_parity_secondary.py", "tests/test_parity_next.py",
                           "tests/test_parity_sweep.py", "tests/test_parity_packed.py",
                           "tests/test_parity_fused_hier.py", "tests/test_parity_fused_lowp.py"],
                          cwd=ROOT, env=checked_env, capture_output=True, text=True,
                          timeout=1800)
    assert proc.returncode == 0, proc.stdout[-4000:] + proc.stderr[-2000:]
    ran = re.search(r"(\d+) passed", proc.stdout)
    assert ran and int(ran.group(1)) >= 60, proc.stdout[-2000:]
    print(proc.stdout.strip().splitlines()[-1])
