"""Oracle: FlowMatch Euler sigma schedule and the Euler update.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Source: Host contract (RGBA-Image-2.1), section 6 "Sampler (FlowMatch Euler,
40 steps, no CFG)", with the scheduler constants of host/scheduler.json:
base_shift 0.5, max_shift 0.9, image sequence lengths 256..8192,
shift_terminal 0.02, 1000 training timesteps.

Reading of "All arrays fp32": the stored arrays (sigmas, timesteps) are float32;
the shift and the terminal stretch are evaluated in float64 and rounded once
at the end. The step in numpy's linspace is (stop - start) / (steps - 1) and the
last entry is set to the end point.
"""
from __future__ import annotations

import math

import numpy as np

BASE_SHIFT = 0.5
MAX_SHIFT = 0.9
BASE_SEQ = 256
MAX_SEQ = 8192
SHIFT_TERMINAL = 0.02
TRAIN_STEPS = 1000


def mu(N: int, base_shift=BASE_SHIFT, max_shift=MAX_SHIFT, base_seq=BASE_SEQ, max_seq=MAX_SEQ) -> float:
    """mu = N*m + b with m = (max - base)/(max_seq - base_seq), b = base - m*base_seq."""
    m = (max_shift - base_shift) / (max_seq - base_seq)
    b = base_shift - m * base_seq
    return N * m + b


def linspace(start: float, stop: float, num: int) -> np.ndarray:
    """numpy.linspace(start, stop, num) in float64, written out: start + i*step, end point exact."""
    if num == 1:
        return np.array([start], dtype=np.float64)
    step = (stop - start) / (num - 1)
    y = np.array([i * step + start for i in range(num)], dtype=np.float64)
    y[-1] = stop
    return y


def flow_sigmas(steps: int, N: int, base_shift=BASE_SHIFT, max_shift=MAX_SHIFT, base_seq=BASE_SEQ,
                max_seq=MAX_SEQ, shift_terminal=SHIFT_TERMINAL, train_steps=TRAIN_STEPS):
    """Return (sigmas float32 [steps+1], timesteps float32 [steps])."""
    s = linspace(1.0, 1.0 / steps, steps)
    e = math.exp(mu(N, base_shift, max_shift, base_seq, max_seq))
    s = e / (e + (1.0 / s - 1.0))                    # exponential time shift
    one_minus = 1.0 - s
    scale = one_minus[-1] / (1.0 - shift_terminal)
    s = 1.0 - one_minus / scale                      # stretch so the last sigma is shift_terminal
    timesteps = (s * train_steps).astype(np.float32)
    sigmas = np.concatenate([s.astype(np.float32), np.zeros(1, np.float32)])
    return sigmas, timesteps


def dit_timestep(timesteps: np.ndarray, i: int) -> np.float32:
    """The DiT's `timestep` input: timesteps[i] / 1000 in float32."""
    return np.float32(np.float32(timesteps[i]) / np.float32(TRAIN_STEPS))


def euler_update(x: np.ndarray, vel: np.ndarray, sigma_i, sigma_next) -> np.ndarray:
    """x + (sigma[i+1] - sigma[i]) * vel in float32, each operation rounded on its own."""
    dt = np.float32(np.float32(sigma_next) - np.float32(sigma_i))
    prod = (np.asarray(vel, np.float32) * dt).astype(np.float32)
    return (np.asarray(x, np.float32) + prod).astype(np.float32)


def cfg_combine(pos: np.ndarray, neg: np.ndarray, g) -> np.ndarray:
    """Classifier-free guidance: neg + g * (pos - neg), float32, each operation rounded.

    Source: MLX page, "Optional modes (approximate or slower)": true CFG uses the
    negative prompt as noise = neg + g * (pos - neg).
    """
    pos = np.asarray(pos, np.float32)
    neg = np.asarray(neg, np.float32)
    d = (pos - neg).astype(np.float32)
    return (neg + (np.float32(g) * d).astype(np.float32)).astype(np.float32)


# ----------------------------------------------------------------------------- DPM++ 2M
#
# MLX page, "Optional modes (approximate or slower)": a DPM++ 2M sampler is offered
# next to FlowMatch Euler; the page gives no formula. Reading: the second-order
# multistep DPM-Solver++ (Lu et al. 2022, "DPM-Solver++: Fast Solver for Guided
# Sampling of Diffusion Probabilistic Models", multistep second-order solver) on the
# flow-matching noise schedule the model is trained on, x_sigma = (1 - sigma) x0 +
# sigma eps, i.e. alpha = 1 - sigma and lambda = log(alpha / sigma). The model's
# data prediction is D = x - sigma v. One step sigma_i -> sigma_{i+1}, h_i =
# lambda_{i+1} - lambda_i:
#     x_{i+1} = (sigma_{i+1} / sigma_i) x_i - alpha_{i+1} (e^{-h_i} - 1) D'
#     D' = (1 + 1/(2 r)) D_i - 1/(2 r) D_{i-1},   r = h_{i-1} / h_i
# With alpha = 1 - sigma, alpha_{i+1} (1 - e^{-h_i}) = 1 - sigma_{i+1}/sigma_i, so
# x_{i+1} = a x_i + (1 - a) D' with a = sigma_{i+1} / sigma_i. The first step (no
# D_{i-1}) and a step whose previous sigma is 1 (lambda = -inf, so 1/(2r) = 0) are
# first order; the last step (sigma_{i+1} = 0, lambda = +inf) returns D_i itself,
# the limit of the first-order step.
#
# Rounding reading (the pages fix none): coefficients are evaluated in float64 from
# the float32 sigmas and rounded once to float32; the element-wise update is float32
# with every operation rounded on its own (no fused multiply-add).

def half_log_snr(sigma) -> float:
    """lambda = log((1 - sigma) / sigma) in float64; -inf at sigma = 1, +inf at 0."""
    s = float(sigma)
    if s >= 1.0:
        return -math.inf
    if s <= 0.0:
        return math.inf
    return math.log1p(-s) - math.log(s)


def dpmpp2m_coeffs(sigmas, i: int):
    """Coefficients of step i: (order, a, b, c0, c1), the four floats in float32.

    order 0: last step, x <- D. order 1: x <- a x + b D. order 2: x <- a x + b (c0 D - c1 D_prev).
    """
    s = float(np.float32(sigmas[i]))
    sn = float(np.float32(sigmas[i + 1]))
    one = np.float32(1.0)
    zero = np.float32(0.0)
    if sn == 0.0:
        return 0, zero, one, one, zero
    a = sn / s
    b = (s - sn) / s
    if i == 0 or float(np.float32(sigmas[i - 1])) >= 1.0:
        return 1, np.float32(a), np.float32(b), one, zero
    lam_prev = half_log_snr(np.float32(sigmas[i - 1]))
    lam = half_log_snr(s)
    lam_next = half_log_snr(sn)
    h = lam_next - lam
    h_prev = lam - lam_prev
    c1 = h / (2.0 * h_prev)          # 1 / (2 r)
    return 2, np.float32(a), np.float32(b), np.float32(1.0 + c1), np.float32(c1)


def dpmpp2m_update(x, vel, d_prev, sigmas, i: int):
    """One DPM++ 2M step in float32. Returns (x_next, D_i); D_i is step i+1's d_prev.

    d_prev is ignored unless the step is second order.
    """
    order, a, b, c0, c1 = dpmpp2m_coeffs(sigmas, i)
    x = np.asarray(x, np.float32)
    sv = (np.float32(sigmas[i]) * np.asarray(vel, np.float32)).astype(np.float32)
    D = (x - sv).astype(np.float32)
    if order == 0:
        return D.copy(), D
    if order == 2:
        Dp = ((c0 * D).astype(np.float32) - (c1 * np.asarray(d_prev, np.float32)).astype(np.float32)).astype(np.float32)
    else:
        Dp = D
    xn = ((a * x).astype(np.float32) + (b * Dp).astype(np.float32)).astype(np.float32)
    return xn, D
