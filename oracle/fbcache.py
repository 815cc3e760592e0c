"""Oracle: the first-block cache ("Fast mode") around the DiT pass.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Source: MLX page, "Optional modes (approximate or slower)": Fast mode is a
first-block cache; block 0 always runs, and blocks 1 to 31 are skipped while
block 0's residual changes less than a threshold (the options table gives
`--first-block-cache 0.08`; the timing table calls the mode approximate).

Readings where the page is silent:
* "block 0's residual" is r0 = x1 - x0 on the image rows, x0 the residual stream
  entering block 0 and x1 the one leaving it (text rows are constant over a run);
* its "change" is the relative mean absolute difference
  sum |r0 - r0_ref| / sum |r0_ref| (float64 sums), and the step is skipped when
  it is strictly below the threshold;
* r0_ref is block 0's residual at the last step that ran every block (not the
  previous step), so a slow drift cannot be skipped indefinitely;
* a skipped step adds the stored residual of blocks 1..31 from that same step,
  x_out = x1 + (x32_ref - x1_ref), then runs the output head as usual;
* a step that sees a new prompt (a joint pass) always runs every block and
  restarts the reference.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from . import dit


@dataclass
class FBCacheState:
    """Reference residuals from the last step that ran every block (image rows)."""
    r0: np.ndarray | None = None      # block 0's residual
    rest: np.ndarray | None = None    # residual of blocks 1..last
    history: list = field(default_factory=list)  # (rel, skipped) per call

    @property
    def valid(self) -> bool:
        return self.r0 is not None


def rel_change(r0: np.ndarray, ref: np.ndarray) -> float:
    """sum |r0 - ref| / sum |ref| in float64; 0 when both sums are 0, inf when only the
    reference is 0."""
    r = np.asarray(r0, np.float64)
    p = np.asarray(ref, np.float64)
    num = float(np.abs(r - p).sum())
    den = float(np.abs(p).sum())
    if den == 0.0:
        return 0.0 if num == 0.0 else math.inf
    return num / den


def decide(state: FBCacheState, r0: np.ndarray, threshold: float, new_prompt: bool):
    """(rel, skip) for this step. rel is inf when there is no usable reference."""
    if new_prompt or not state.valid or state.r0.shape != r0.shape:
        return math.inf, False
    rel = rel_change(r0, state.r0)
    return rel, rel < threshold


def dit_forward_fbcache(weights, img_tokens, txt_feats, t, txt_cos, txt_sin, img_cos, img_sin,
                        state: FBCacheState, threshold: float, new_prompt: bool, nblocks: int = None):
    """One DiT pass under the first-block cache. Returns (vel [N, 64], rel, skipped).

    Every pass here recomputes the text rows (their K/V are constant over a run, so
    this equals reading a capture); only the image rows enter r0 and the cache.
    """
    g = weights.glob
    heads = weights.dims.heads
    L = txt_feats.shape[0]
    N = img_tokens.shape[0]
    R = L + N
    mods = dit.row_mods(dit.modulation(g, t), dit.modulation(g, 0.0), L, R)
    cos = np.concatenate([txt_cos, img_cos], axis=0)
    sin = np.concatenate([txt_sin, img_sin], axis=0)
    nb = weights.nblocks if nblocks is None else nblocks

    x0 = dit.embed(g, img_tokens, txt_feats)
    x1 = dit.block_forward(weights.block(0), x0, mods, L, cos, sin, heads)
    r0 = (x1[L:] - x0[L:]).astype(np.float32)
    rel, skip = decide(state, r0, threshold, new_prompt)
    if skip:
        x_img = (x1[L:] + state.rest).astype(np.float32)
    else:
        x = x1
        for b in range(1, nb):
            x = dit.block_forward(weights.block(b), x, mods, L, cos, sin, heads)
        x_img = x[L:]
        state.r0 = r0
        state.rest = (x[L:] - x1[L:]).astype(np.float32)
    state.history.append((rel, skip))
    return dit.head(g, x_img), rel, skip
