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



WAIT_CHILD = r"""
import time
import torch
from zero_distributed_optimizer_gb300 import binding as B
from zero_distributed_optimizer_gb300 import workloads as W

assert B.LIB_PATH.endswith("libdopt_checked.so"), B.LIB_PATH
D = 4
L = B.dopt_build_range_map([130, 260, 90, 310, 210], D, 0, 1).to_device()  # one tile
N = L.padded_numel
master, m, v, params, grads = W.random_case(N, D, 1, "bf16", seed=7)
state = [x.cuda() for x in (master, m, v)]
params = [p.cuda() for p in params]
grads = [g.cuda() for g in grads[0]]
adam = B.AdamConfig(grad_scale=1.0 / D)
before = [x.clone() for x in state + params]
B.stage_timeouts(reset=True)
B.stage_wait_test(16)  # 16 bytes that no copy delivers
t0 = time.monotonic()
B.dopt_step(L, adam, 1, grads, *state, params, stage=True)
torch.cuda.synchronize()
waited = time.monotonic() - t0
B.stage_wait_test(0)
assert B.stage_timeouts() == 1, B.stage_timeouts()  # the tile's one CTA
assert 3.5 < waited < 60, waited  # its two bounded waits of 2 s each ran out
for x, y in zip(state + params, before):  # the tile was left alone
    assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                       y.view(torch.int16) if y.dtype == torch.bfloat16 else y)
# the context is still usable: the same step staged and direct, bit for bit
direct = [x.clone() for x in before]
B.dopt_step(L, adam, 1, grads, *state, params, stage=True)
B.dopt_step(L, adam, 1, grads, *direct[:3], direct[3:])
torch.cuda.synchronize()
for x, y in zip(state + params, direct):
    assert torch.equal(x.view(torch.int32) if x.dtype == torch.float32 else x.view(torch.int16),
                       y.view(torch.int32) if y.dtype == torch.float32 else y.view(torch.int16))
assert not torch.equal(state[0], before[0])
assert B.stage_timeouts(reset=True) == 1  # no further CTA ran out
print("WAIT_OK")
"""


def test_staged_wait_runs_out_without_fault():
    """The staged step's bounded copy wait, made to run out in the test
    build (the CTA's mbarrier expects 16 bytes that no copy delivers): the
    call returns, the CTA is counted and leaves its tile untouched, and the
    next steps on the same context give the direct path's results."""
    from zero_distributed_optimizer_gb300 import build

    build.build(checked=True)
    env = dict(os.environ, DOPT_CHECKED="1")
    r = subprocess.run([sys.executable, "-c", WAIT_CHILD], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "WAIT_OK" in r.stdout
