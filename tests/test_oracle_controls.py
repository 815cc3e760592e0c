"""Controls: mistakes planted in the oracle (on the CPU) must break its pins.

Each control swaps one oracle function for a plausible wrong version and checks
that the vectorised block no longer matches the independent row-loop form.
"""
import numpy as np
import pytest

import synth
from oracle import attention, dit, rope

TINY = synth.TINY


def _case():
    W = synth.Weights(seed=5, dims=TINY)
    L, h, w = 3, 2, 2
    R = L + h * w
    tc, ts, ic, is_ = rope.token_tables(L, h, w, axes=TINY.axes)
    cos, sin = np.concatenate([tc, ic]), np.concatenate([ts, is_])
    mods = dit.row_mods(dit.modulation(W.glob, 0.37), dit.modulation(W.glob, 0.0), L, R)
    x = synth.input_f32(5, 0, (R, TINY.hidden))
    ref = dit.block_forward_rowloop(W.block(0), x, mods, L, cos, sin, TINY.heads)
    return W, x, mods, L, cos, sin, ref


def _half_split_rope(x, cos, sin):
    half = x.shape[-1] // 2
    a, b = x[..., :half], x[..., half:]
    c, s = cos[:, None, :], sin[:, None, :]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1).astype(np.float32)


def _no_causal(q, k, v, L, q_chunk=2048):
    return attention.attention_masked(q, k, v, 0, q_chunk)


def _swapped_chunks(mod_row):
    H = mod_row.shape[-1] // 4
    return mod_row[..., H:2 * H], mod_row[..., 0:H], mod_row[..., 2 * H:3 * H], mod_row[..., 3 * H:4 * H]


def _rms_without_eps(x, eps=0.0):
    x = np.asarray(x, np.float32)
    return (x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True))).astype(np.float32) * np.float32(1.01)


CONTROLS = {
    "rope_half_split": ("rope", _half_split_rope),
    "text_sees_image": ("attention_masked", _no_causal),
    "mod_chunks_swapped": ("mod_chunks", _swapped_chunks),
    "norm_scaled": ("rmsnorm", _rms_without_eps),
}


@pytest.mark.parametrize("name", sorted(CONTROLS))
def test_control_is_red(name, monkeypatch):
    W, x, mods, L, cos, sin, ref = _case()
    attr, bad = CONTROLS[name]
    monkeypatch.setattr(dit, attr, bad)
    got = dit.block_forward(W.block(0), x, mods, L, cos, sin, TINY.heads)
    err = np.abs(got - ref).max() / np.abs(ref - x).max()
    # the pin in test_oracle_dit.py accepts err <= 2e-5; a control must land far outside it
    assert err > 2e-4, f"control {name} went unnoticed (err {err:.2e})"


def test_controls_green_without_plant():
    W, x, mods, L, cos, sin, ref = _case()
    got = dit.block_forward(W.block(0), x, mods, L, cos, sin, TINY.heads)
    assert np.abs(got - ref).max() / np.abs(ref - x).max() < 2e-5
