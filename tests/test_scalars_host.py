"""The library evaluates beta^t by repeated squaring in double (the same
multiplies on the host for dopt_step and on the device for
dopt_step_counted), where the oracle calls pow.  The float scalars
lr / (1 - beta1^t) and sqrt(1 - beta2^t) they lead to must be the same.
The squaring is restated here in Python floats (IEEE double, one rounding
per multiply) and compared with the oracle's scalars."""
import math

import numpy as np
import pytest

import oracle
from zero_distributed_optimizer_gb300 import workloads as W


def beta_pow(b: float, t: int) -> float:
    r, x = 1.0, b
    while t > 0:
        if t & 1:
            r = r * x
        t >>= 1
        if t > 0:
            x = x * x
    return r


def _adams():
    seen = []
    for w in (W.toy_1000(), W.gpt2_small(), W.llama_1p3b(), W.sweep_256m(8, 64),
              W.moe_many_small()):
        seen.append(w.adam_kwargs())
    seen += [dict(lr=3e-3, beta1=0.85, beta2=0.97), dict(lr=1e-4, beta1=0.9, beta2=0.999),
             dict(lr=0.1, beta1=0.5, beta2=0.99), dict(lr=1e-3, beta1=0.0, beta2=0.0)]
    return seen


@pytest.mark.parametrize("kw", _adams())
def test_squaring_gives_the_oracles_scalars(kw):
    adam = oracle.make_adam(**kw)
    lr, b1, b2 = (float(np.float32(kw.get(k, d))) for k, d in
                  (("lr", 1e-3), ("beta1", 0.9), ("beta2", 0.95)))
    rng = np.random.default_rng(5)
    ts = list(range(1, 5001)) + [int(x) for x in rng.integers(5001, 1 << 62, 300)] + [1 << 62]
    for t in ts:
        want = oracle.step_scalars(adam, t)
        step_size = np.float32(lr / (1.0 - beta_pow(b1, t)))
        bc2_sqrt = np.float32(math.sqrt(1.0 - beta_pow(b2, t)))
        assert step_size == np.float32(want["step_size"]), t
        assert bc2_sqrt == np.float32(want["bc2_sqrt"]), t
