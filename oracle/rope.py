"""Oracle: 3-axis RoPE tables, token positions and noise packing.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this module;
only tests/, the smoke check and the bench's CPU-baseline leg use it.

Sources
-------
* Host contract (RGBA-Image-2.1, Core AI port of Qwen-Image-2.1), section 4
  "Sequence layout and RoPE": positions of text and image tokens, the per-axis
  tables over positions -1024..8191 with widths (16, 56, 56), and the way a
  token's 64 columns are the three axis rows concatenated.
* Same page, section 5 "Noise and pack": x[0, y*w + x, c] = z[c, y, x].

Rounding reading (the page names torch.polar in float32 but fixes no rounding):
    omega_k = fl32(theta ** (-2k/d))            evaluated in float64
    angle   = fl32(fl32(pos) * omega_k)          one float32 multiply
    value   = fl32(cos(angle)), fl32(sin(angle)) cos/sin evaluated in float64
Each step is a correctly rounded float32 result of a float64 value, so it has a
single right answer.
"""
from __future__ import annotations

import numpy as np

POS_LO = -1024
POS_HI = 8191
NPOS = POS_HI - POS_LO + 1  # 9216 rows


def axis_freqs(d: int, theta: float = 10000.0) -> np.ndarray:
    """omega_k = 1 / theta^(2k/d) for k < d/2, as float32 (host contract section 4)."""
    k = np.arange(d // 2, dtype=np.float64)
    return np.array([np.float32(float(theta) ** (-(2.0 * kk) / d)) for kk in k], dtype=np.float32)


def axis_table(d: int, theta: float = 10000.0):
    """(cos, sin) float32 [9216, d/2]; row p + 1024 holds position p."""
    pos = np.arange(POS_LO, POS_HI + 1, dtype=np.float32)
    w = axis_freqs(d, theta)
    angle = (pos[:, None] * w[None, :]).astype(np.float32)  # one fp32 multiply per entry
    a64 = angle.astype(np.float64)
    return np.cos(a64).astype(np.float32), np.sin(a64).astype(np.float32)


def axis_tables(axes=(16, 56, 56), theta: float = 10000.0):
    return [axis_table(d, theta) for d in axes]


def text_positions(L: int) -> np.ndarray:
    """Text token i -> (i, i, i)."""
    i = np.arange(L, dtype=np.int64)
    return np.stack([i, i, i], axis=1)


def image_positions(L: int, h: int, w: int) -> np.ndarray:
    """Image token (y, x), index y*w + x -> (L, y - (h - h//2), x - (w - w//2))."""
    y, x = np.meshgrid(np.arange(h), np.arange(w), indexing="ij")
    y = y.reshape(-1)
    x = x.reshape(-1)
    f = np.full_like(y, L)
    return np.stack([f, y - (h - h // 2), x - (w - w // 2)], axis=1).astype(np.int64)


def gather(tables, pos: np.ndarray):
    """Concatenate the three axis rows for each token: [T, sum(d/2)] cos and sin."""
    cos = np.concatenate([tables[a][0][pos[:, a] - POS_LO] for a in range(3)], axis=1)
    sin = np.concatenate([tables[a][1][pos[:, a] - POS_LO] for a in range(3)], axis=1)
    return cos.astype(np.float32), sin.astype(np.float32)


def token_tables(L: int, h: int, w: int, axes=(16, 56, 56), theta: float = 10000.0):
    """txt_cos, txt_sin [L, 64] and img_cos, img_sin [h*w, 64] for one image."""
    tabs = axis_tables(axes, theta)
    tc, ts = gather(tabs, text_positions(L))
    ic, is_ = gather(tabs, image_positions(L, h, w))
    return tc, ts, ic, is_


def pack_noise(z: np.ndarray) -> np.ndarray:
    """Channel-major latent z[c, y, x] -> tokens x[y*w + x, c] (host contract section 5)."""
    c, h, w = z.shape
    out = np.empty((h * w, c), dtype=z.dtype)
    for yy in range(h):
        for xx in range(w):
            out[yy * w + xx, :] = z[:, yy, xx]
    return out
