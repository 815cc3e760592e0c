"""Pins for oracle/sched.py: numbers the pages print, closed forms, invariants."""
import math
import os

import numpy as np
import pytest

from oracle import sched

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sched_pins.txt")


def _golden():
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line.split()


def _digits(x, n):
    return math.floor(x * 10 ** n + 1e-9) / 10 ** n


def test_pages_printed_values():
    seen = 0
    for kind, N, val, digits in _golden():
        N, digits = int(N), int(digits)
        if kind == "mu":
            got = sched.mu(N)
            # the pages print either a rounded value or a truncated prefix ("0.5387...")
            assert float(val) in (round(got, digits), _digits(got, digits))
        elif kind == "sigma1":
            s, _ = sched.flow_sigmas(40, N)
            assert round(float(s[1]), digits) == float(val)
            assert abs(float(s[1]) - 0.975) > 0.009  # not the plain linspace value
        seen += 1
    assert seen == 5


def test_end_points():
    for N in (256, 576, 1024, 4096, 16384):
        s, ts = sched.flow_sigmas(40, N)
        assert s.dtype == np.float32 and s.shape == (41,) and ts.shape == (40,)
        assert s[0] == np.float32(1.0)
        assert s[39] == np.float32(0.02)   # shift_terminal
        assert s[40] == 0.0
        assert (np.diff(s) < 0).all()


def test_against_high_precision():
    """The float32 sigmas are the exact schedule rounded once (plus float64 error)."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.prec = 100
    for N in (256, 4096, 16384):
        s, ts = sched.flow_sigmas(40, N)
        m = mpmath.mpf(0.4) / mpmath.mpf(8192 - 256)
        mu = N * m + (mpmath.mpf(0.5) - 256 * m)
        e = mpmath.exp(mu)
        lin = [1 + i * (mpmath.mpf(1) / 40 - 1) / 39 for i in range(40)]
        sh = [e / (e + (1 / x - 1)) for x in lin]
        scale = (1 - sh[-1]) / (1 - mpmath.mpf("0.02"))
        exact = [1 - (1 - x) / scale for x in sh]
        for i in range(40):
            ref = float(exact[i])
            # within one float32 ulp of the exact value
            assert abs(float(s[i]) - ref) <= np.spacing(np.float32(ref)), (N, i)
            assert abs(float(ts[i]) - 1000 * ref) <= np.spacing(np.float32(1000 * ref)), (N, i)


def test_shift_is_a_logit_offset():
    """Before the terminal stretch, logit(sigma') = mu + logit(sigma)."""
    N = 1024
    mu = sched.mu(N)
    s = sched.linspace(1.0, 1 / 40, 40)[1:]
    e = math.exp(mu)
    sh = e / (e + (1.0 / s - 1.0))
    lhs = np.log(sh / (1 - sh))
    rhs = mu + np.log(s / (1 - s))
    assert np.allclose(lhs, rhs, rtol=0, atol=1e-12)


def test_linspace_matches_numpy():
    for n in (2, 5, 25, 40):
        assert (sched.linspace(1.0, 1.0 / n, n) == np.linspace(1.0, 1.0 / n, n)).all()


def test_dit_timestep_multiply_then_divide():
    s, ts = sched.flow_sigmas(40, 256)
    for i in range(40):
        t = sched.dit_timestep(ts, i)
        assert t == np.float32(ts[i] / np.float32(1000.0))
        assert abs(float(t) - float(s[i])) < 1e-6


def test_euler_closed_form_and_rounding():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(1000).astype(np.float32)
    v = rng.standard_normal(1000).astype(np.float32)
    y = sched.euler_update(x, v, np.float32(0.9), np.float32(0.85))
    dt = np.float32(np.float32(0.85) - np.float32(0.9))
    for i in range(0, 1000, 37):
        # separately rounded product and sum, checked in float64 with explicit rounding
        p = np.float32(float(v[i]) * float(dt))
        assert y[i] == np.float32(float(x[i]) + float(p))


def test_euler_telescopes():
    """With a constant velocity c the 40 updates move x by c * (sigma_40 - sigma_0) = -c."""
    s, _ = sched.flow_sigmas(40, 4096)
    x = np.zeros(4, np.float32)
    c = np.array([1.0, -2.0, 0.5, 3.0], np.float32)
    for i in range(40):
        x = sched.euler_update(x, c, s[i], s[i + 1])
    assert np.allclose(x, -c, rtol=0, atol=1e-5)


def test_cfg_combine_closed_forms():
    rng = np.random.default_rng(4)
    pos = rng.standard_normal(500).astype(np.float32)
    neg = rng.standard_normal(500).astype(np.float32)
    # g = 0 returns the negative branch exactly; g = 1 the conditional one to within rounding
    assert np.array_equal(sched.cfg_combine(pos, neg, 0.0), neg)
    assert np.allclose(sched.cfg_combine(pos, neg, 1.0), pos, rtol=0, atol=1e-6)
    # equal branches are a fixed point for any g
    assert np.array_equal(sched.cfg_combine(pos, pos, 4.5), pos)
    # affine in g: the midpoint of g = 1 and g = 3 is g = 2
    a, b, c = (sched.cfg_combine(pos, neg, gg).astype(np.float64) for gg in (1.0, 2.0, 3.0))
    assert np.allclose((a + c) / 2, b, rtol=0, atol=1e-5)
    # the stated order of operations, element by element in float64 with explicit rounding
    for i in range(0, 500, 53):
        d = np.float32(float(pos[i]) - float(neg[i]))
        m = np.float32(float(np.float32(2.5)) * float(d))
        assert sched.cfg_combine(pos[i:i + 1], neg[i:i + 1], 2.5)[0] == np.float32(float(neg[i]) + float(m))
