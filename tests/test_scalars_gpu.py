"""The two step-dependent Adam scalars, step_size = lr / (1 - beta1^t) and
bc2_sqrt = sqrt(1 - beta2^t), against the oracle, over seeded random
hyper-parameters and step numbers.

Both sides evaluate them in double and round to float once.  The oracle
takes beta^t from C's pow.  The host entry points (dopt_step) call the same
pow, so every step they take must equal the oracle's bit for bit, whatever
the hyper-parameters.  The counted steps evaluate the scalars on the device
(binary powering with an error bound, and an exact double-double fallback
when the bound leaves the float open): their scalars, read back from the
counter, must equal the oracle's too.  The last test takes (beta, t) pairs
where binary powering alone rounds to another float than pow does (found
by a CPU search over float betas), so the fallback has to run there."""
from dataclasses import asdict

import numpy as np
import pytest
import torch

import oracle
from parity import assert_bf16_close, assert_f32_close, t2np_bf16, t2np_f32, t2np_grad
from zero_distributed_optimizer_gb300 import binding as B
from zero_distributed_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def random_adams(n, seed):
    """n seeded AdamW hyper-parameter sets over the valid ranges, with the
    betas spread from 0 to just below 1 (where the bias corrections change
    slowly and binary powering's error is amplified most)."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        lr = float(10.0 ** rng.uniform(-6, 0))
        b1 = float(1.0 - 10.0 ** rng.uniform(-6.5, 0)) if i % 7 else 0.0
        b2 = float(1.0 - 10.0 ** rng.uniform(-7, -0.3))
        eps = float(10.0 ** rng.uniform(-12, -4))
        wd = float(rng.uniform(0.0, 0.3))
        out.append(B.AdamConfig(lr=lr, beta1=min(b1, 0.99999994), beta2=min(b2, 0.99999994),
                                eps=eps, weight_decay=wd, grad_scale=0.5))
    return out


def _f32_bits(x):
    return int(np.float32(x).view(np.uint32))


def test_host_steps_match_oracle_for_random_hyperparameters():
    """dopt_step under 150 random hyper-parameter sets at step numbers from
    1 to 10^6: every element of master/m/v and of both param replicas equals
    the oracle's after every step."""
    sizes, wd, D = [100, 37, 500, 3], [1, 0, 1, 0], 2
    L = B.dopt_build_range_map(sizes, D, 0, 1, wd).to_device()
    N = L.padded_numel
    ts = (1, 2, 3, 5, 17, 301, 4097, 999_983)
    not_exact = 0
    for i, adam in enumerate(random_adams(150, seed=31)):
        master, m, v, params, grads = W.random_case(N, D, len(ts), "bf16", seed=900 + i)
        hs = [master.numpy().copy(), m.numpy().copy(), v.numpy().copy()]
        hp = [t2np_bf16(p).copy() for p in params]
        ds = [master.to(DEV), m.to(DEV), v.to(DEV)]
        dp = [p.to(DEV) for p in params]
        oadam = oracle.make_adam(**asdict(adam))
        for k, t in enumerate(ts):
            B.dopt_step(L, adam, t, [g.to(DEV) for g in grads[k]], *ds, dp)
            oracle.step(sizes, wd, D, 0, 1, oadam, t, [t2np_grad(g) for g in grads[k]], *hs, hp)
            torch.cuda.synchronize()
            for name, x, y in zip(("master", "exp_avg", "exp_avg_sq"), ds, hs):
                not_exact += assert_f32_close(t2np_f32(x), y, f"{name} set {i} t {t}")
            for r in range(D):
                not_exact += assert_bf16_close(t2np_bf16(dp[r]), hp[r], f"param{r} set {i} t {t}")
    assert not_exact == 0


def _counted_scalars(L, adam, counter, t, state, params, grads):
    counter[0] = t
    B.dopt_step_counted(L, adam, counter, grads, *state, params)
    return B.counter_scalars(counter)


def _tiny_case():
    L = B.dopt_build_range_map([16], 1, 0, 1).to_device()
    master, m, v, params, grads = W.random_case(L.padded_numel, 1, 1, "bf16", seed=3)
    return L, [master.to(DEV), m.to(DEV), v.to(DEV)], [params[0].to(DEV)], \
        [grads[0][0].to(DEV)]


def test_counted_scalars_match_oracle_for_random_hyperparameters():
    """The counted step's scalars under 200 random hyper-parameter sets at 40
    step numbers each (the first 24, then spread up to 2^62): bit for bit
    the oracle's, and never left undecided."""
    L, state, params, grads = _tiny_case()
    rng = np.random.default_rng(77)
    ts = list(range(1, 25)) + sorted({int(x) for x in 10 ** rng.uniform(1.5, 7, 12)}) + \
        [1 << 40, (1 << 62) - 1, 1 << 62]
    counter = B.step_counter(1, DEV)
    checked = 0
    for i, adam in enumerate(random_adams(200, seed=5)):
        oadam = oracle.make_adam(**asdict(adam))
        for t in ts:
            got = _counted_scalars(L, adam, counter, t, state, params, grads)
            want = oracle.step_scalars(oadam, t)
            assert _f32_bits(got[0]) == _f32_bits(want["step_size"]), (i, t, adam, got, want)
            assert _f32_bits(got[1]) == _f32_bits(want["bc2_sqrt"]), (i, t, adam, got, want)
            checked += 1
    assert B.counter_state(counter) == (ts[-1] + 1, 0)
    exact, undecided = B.counter_diagnostics(counter)
    assert undecided == 0
    assert checked == 200 * len(ts)


# (beta1, beta2, t): binary powering alone rounds step_size (beta1) or
# bc2_sqrt (beta2) to a float next to pow's; found by a CPU search over the
# float betas in [0.8, 1) and [0.99, 1), lr = 1e-3.  The other beta is 0.9 /
# 0.95, whose scalars are unambiguous at these t.
POWERING_DIFFERS = [
    (0.9, 0.9999985694885254, 6),
    (0.9, 0.9999995231628418, 18),
    (0.9, 0.9935411810874939, 302),
    (0.9, 0.9998261332511902, 3064),
    (0.9989400506019592, 0.95, 159),
    (0.9995810389518738, 0.95, 242),
    (0.9998176693916321, 0.95, 371),
    (0.9999927282333374, 0.95, 3767),
]


@pytest.mark.parametrize("b1,b2,t", POWERING_DIFFERS)
def test_counted_scalars_where_powering_alone_would_differ(b1, b2, t):
    """At these (beta, t) the fast evaluation cannot decide, the exact one
    runs (the counter counts it) and the scalars are still the oracle's; a
    dopt_step at the same t gives the counted step's result bit for bit."""
    L, state, params, grads = _tiny_case()
    adam = B.AdamConfig(lr=1e-3, beta1=b1, beta2=b2)
    counter = B.step_counter(1, DEV)
    ref_state = [x.clone() for x in state]
    ref_params = [p.clone() for p in params]
    got = _counted_scalars(L, adam, counter, t, state, params, grads)
    want = oracle.step_scalars(oracle.make_adam(**asdict(adam)), t)
    assert _f32_bits(got[0]) == _f32_bits(want["step_size"]), (got, want)
    assert _f32_bits(got[1]) == _f32_bits(want["bc2_sqrt"]), (got, want)
    assert B.counter_diagnostics(counter) == (1, 0)
    B.dopt_step(L, adam, t, grads, *ref_state, ref_params)
    torch.cuda.synchronize()
    for x, y in zip(state + params, ref_state + ref_params):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
