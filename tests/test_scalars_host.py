"""The argument behind the counted steps' device scalars, checked on the CPU.

The host entry points take beta^t from C's pow, like the oracle.  The
counter kernel cannot: it computes beta^t by binary powering, whose result p
is within (t - 1) * 2^-53 (relative) of the exact power, bounds pow's double
by [p - B, p + B] with B = p * (t + 2) * 2^-52 + 2^-1000, and accepts a
scalar when both ends of that interval round to the same float (the scalars
are monotone in beta^t).  This restates that check in Python's IEEE doubles
(numpy, one rounding per operation, as on the device) and checks on seeded
random draws that an accepted float is always pow's float, and that the
(beta, t) pairs the GPU test uses for the exact fallback are ones where
binary powering alone rounds to another float than pow."""
import math

import numpy as np
import pytest

import oracle

LR = float(np.float32(1e-3))


def powering(b, t):
    """beta^t by binary powering, elementwise over an array of doubles."""
    r = np.ones_like(b)
    x = b.copy()
    while t > 0:
        if t & 1:
            r = r * x
        t >>= 1
        if t > 0:
            x = x * x
    return r


def scalar(which, p):
    d = 1.0 - p
    return (LR / d).astype(np.float32) if which == 0 else np.sqrt(d).astype(np.float32)


@pytest.mark.parametrize("which,lo", [(0, 0.5), (0, 0.99), (1, 0.9), (1, 0.999)])
@pytest.mark.parametrize("t", [2, 3, 7, 31, 100, 1000, 4097])
def test_accepted_interval_float_is_pows_float(which, lo, t):
    rng = np.random.default_rng(1000 * t + int(lo * 1000) + which)
    b = rng.uniform(lo, 1.0, 200_000).astype(np.float32).astype(np.float64)
    b = b[b < 1.0]
    p = powering(b, t)
    bound = p * (t + 2.0) * 2.0 ** -52 + 2.0 ** -1000
    lo_end = scalar(which, np.maximum(p - bound, 0.0))
    hi_end = scalar(which, p + bound)
    want = scalar(which, np.power(b, float(t)))  # C's pow, elementwise
    accepted = lo_end == hi_end
    assert accepted.mean() > 0.99
    assert np.array_equal(lo_end[accepted], want[accepted])


@pytest.mark.parametrize("b1,b2,t", [
    (0.9, 0.9999985694885254, 6), (0.9, 0.9999995231628418, 18),
    (0.9, 0.9935411810874939, 302), (0.9, 0.9998261332511902, 3064),
    (0.9989400506019592, 0.95, 159), (0.9995810389518738, 0.95, 242),
    (0.9998176693916321, 0.95, 371), (0.9999927282333374, 0.95, 3767)])
def test_fallback_cases_are_where_powering_alone_differs(b1, b2, t):
    which, b = (1, b2) if b1 == 0.9 else (0, b1)
    assert float(np.float32(b)) == b
    p = float(powering(np.array([b]), t)[0])
    assert scalar(which, np.array([p]))[0] != scalar(which, np.array([math.pow(b, t)]))[0]
    # and the oracle's scalar is pow's
    s = oracle.step_scalars(oracle.make_adam(lr=1e-3, beta1=b1, beta2=b2), t)
    got = s["step_size"] if which == 0 else s["bc2_sqrt"]
    assert np.float32(got) == scalar(which, np.array([math.pow(b, t)]))[0]
