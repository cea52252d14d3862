"""The test build with the kernels' device-side index checks
(libdopt_checked.so, DOPT_DEVICE_CHECKS): stepping valid layouts through
every kernel fails no check, and the checked build gives the same results
as the oracle.  Run in a child process so that the binding loads the
checked library."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path.insert(0, "tests")
import torch
import test_straddle_gpu as S
import test_instances_gpu as I
import test_allreduce_buckets_gpu as A
from zero_distributed_optimizer_gb300 import binding as B

assert B.LIB_PATH.endswith("libdopt_checked.so"), B.LIB_PATH
B.device_checks(reset=True)
for case in range(len(S.CASES)):
    for gather in (True, False):
        S.test_straddling_step(case, gather)
    S.test_straddling_counted_and_allreduce_steps(case)
    S.test_straddling_clipped_step(case)
for case in range(len(I.CASES)):
    I.test_instances_gather_kernel(case)
    I.test_instances_allreduce_and_clipped(case)
for case in range(len(A.CASES)):
    A.test_bucket_launches_equal_whole_step(case, 3)
A.test_bucket_range_launch_covers_only_its_buckets()
torch.cuda.synchronize()
flags, first = B.device_checks()
assert flags == 0 and first == -1, (flags, first)
print("CHECKS_OK")
"""


def test_checked_build_passes_every_check():
    from zero_distributed_optimizer_gb300 import build

    build.build(checked=True)
    env = dict(os.environ, DOPT_CHECKED="1")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "CHECKS_OK" in r.stdout

