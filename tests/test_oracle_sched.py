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


# ----------------------------------------------------------------------------- DPM++ 2M

def _gaussian_velocity(m, s):
    """Exact flow-matching velocity when every coordinate of x0 is N(m, s^2):
    D(x, sigma) = E[x0 | x_sigma = x] in closed form, v = (x - D) / sigma."""
    def vel(x, sg):
        sg = float(sg)
        gain = (1 - sg) * s * s / ((1 - sg) ** 2 * s * s + sg * sg)
        D = m + gain * (x.astype(np.float64) - (1 - sg) * m)
        return ((x - D) / sg).astype(np.float32)
    return vel


def test_dpmpp2m_point_mass_stays_on_the_path():
    """With all data at one point x0, v = (x - x0) / sigma and D = x0 at every step: the
    exponential integrator is then exact, so x stays on (1 - sigma) x0 + sigma eps and
    the last step lands on x0."""
    rng = np.random.default_rng(7)
    x0 = rng.standard_normal(4096).astype(np.float32)
    eps = rng.standard_normal(4096).astype(np.float32)
    sig, _ = sched.flow_sigmas(40, 4096)
    x, dp = eps.copy(), None
    for i in range(40):
        v = ((x.astype(np.float64) - x0) / float(sig[i])).astype(np.float32)
        x, dp = sched.dpmpp2m_update(x, v, dp, sig, i)
        s = float(sig[i + 1])
        on_path = (1 - s) * x0.astype(np.float64) + s * eps.astype(np.float64)
        assert np.abs(x - on_path).max() < 2e-5, i
    assert np.abs(x - x0).max() < 2e-6


def test_dpmpp2m_first_order_step_is_euler():
    """alpha = 1 - sigma makes the first-order step x + (sigma_{i+1} - sigma_i) v."""
    rng = np.random.default_rng(8)
    x = rng.standard_normal(1 << 14).astype(np.float32)
    v = rng.standard_normal(1 << 14).astype(np.float32)
    sig, _ = sched.flow_sigmas(40, 1024)
    order, a, b, c0, c1 = sched.dpmpp2m_coeffs(sig, 0)
    assert order == 1 and abs(float(a) + float(b) - 1.0) < 1e-7
    got, D = sched.dpmpp2m_update(x, v, None, sig, 0)
    ref = x.astype(np.float64) + (float(sig[1]) - float(sig[0])) * v.astype(np.float64)
    assert np.abs(got - ref).max() < 4e-6 * (1 + np.abs(ref).max())
    assert np.array_equal(D, (x - (sig[0] * v).astype(np.float32)).astype(np.float32))


def test_dpmpp2m_correction_is_the_lambda_midpoint():
    """The 2M data estimate extrapolates D linearly in lambda through the last two
    evaluations to the middle of the step, lambda_i + h_i / 2."""
    sig, _ = sched.flow_sigmas(40, 4096)
    for i in (2, 5, 17, 38):
        order, a, b, c0, c1 = sched.dpmpp2m_coeffs(sig, i)
        assert order == 2
        lp, l0, ln = (sched.half_log_snr(sig[j]) for j in (i - 1, i, i + 1))
        A, B = 0.3, -1.7                           # D(lambda) = A + B lambda
        D_prev, D_i = A + B * lp, A + B * l0
        mid = A + B * (l0 + (ln - l0) / 2)
        assert abs(float(c0) * D_i - float(c1) * D_prev - mid) < 1e-6 * (1 + abs(mid))
        assert abs(float(c0) - 1.0 - float(c1)) <= np.spacing(np.float32(c0))  # each rounded once from float64


def test_dpmpp2m_is_second_order():
    """Gaussian data (exact ODE solution known): the error at sigma = 0.02 falls ~4x per
    doubling of the step count; Euler's falls ~2x."""
    m, s = 0.7, 1.3
    vel = _gaussian_velocity(m, s)
    z = np.random.default_rng(0).standard_normal(20000).astype(np.float32)

    def err(steps, dpm):
        sig, _ = sched.flow_sigmas(steps, 4096)
        sig = sig[:-1]                             # stop at the terminal sigma 0.02
        x, dp = z.copy(), None
        for i in range(len(sig) - 1):
            v = vel(x, sig[i])
            if dpm:
                x, dp = sched.dpmpp2m_update(x, v, dp, sig, i)
            else:
                x = sched.euler_update(x, v, sig[i], sig[i + 1])
        se = float(sig[-1])
        exact = (1 - se) * m + math.sqrt((1 - se) ** 2 * s * s + se * se) * z.astype(np.float64)
        return np.abs(x - exact).max()

    e = [err(n, True) for n in (20, 40, 80)]
    for k in range(2):
        assert 3.6 < e[k] / e[k + 1] < 6.0, e
    eu = [err(n, False) for n in (40, 80)]
    assert 1.8 < eu[0] / eu[1] < 2.2 and e[1] < eu[0] / 4


def test_dpmpp2m_step_kinds():
    sig, _ = sched.flow_sigmas(40, 4096)
    assert sched.dpmpp2m_coeffs(sig, 0)[0] == 1            # no previous D
    assert sched.dpmpp2m_coeffs(sig, 1)[0] == 1            # previous sigma is 1: lambda = -inf
    assert sched.dpmpp2m_coeffs(sig, 2)[0] == 2
    assert sched.dpmpp2m_coeffs(sig, 39)[0] == 0           # sigma_40 = 0
    x = np.array([1.0, -2.0, 3.0], np.float32)
    v = np.array([0.5, 0.25, -1.0], np.float32)
    xn, D = sched.dpmpp2m_update(x, v, None, sig, 39)
    assert np.array_equal(xn, D) and np.array_equal(D, (x - (sig[39] * v).astype(np.float32)).astype(np.float32))
    # a schedule that does not start at 1 still takes a first-order first step
    s2 = np.array([0.9, 0.5, 0.2, 0.0], np.float32)
    assert [sched.dpmpp2m_coeffs(s2, i)[0] for i in range(3)] == [1, 2, 0]
    assert sched.half_log_snr(1.0) == -math.inf and sched.half_log_snr(0.0) == math.inf
    assert sched.half_log_snr(0.5) == 0.0


def test_dpmpp2m_midpoint_pin_rejects_an_inverted_ratio():
    """Control: 1/(2r) written with r inverted (h_i / h_{i-1} in place of h_{i-1} / h_i)
    still converges at second order, so only the midpoint pin can catch it."""
    sig, _ = sched.flow_sigmas(40, 4096)
    i = 5
    lp, l0, ln = (sched.half_log_snr(sig[j]) for j in (i - 1, i, i + 1))
    wrong_c1 = (l0 - lp) / (2 * (ln - l0))
    A, B = 0.3, -1.7
    D_prev, D_i = A + B * lp, A + B * l0
    mid = A + B * (l0 + (ln - l0) / 2)
    assert abs((1 + wrong_c1) * D_i - wrong_c1 * D_prev - mid) > 1e-3
