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
