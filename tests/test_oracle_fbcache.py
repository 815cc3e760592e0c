"""Pins for oracle/fbcache.py: the first-block cache around the DiT pass.

Closed forms and special cases: threshold 0 is the plain pass bit for bit; a
repeated input has zero change and a skipped pass reproduces the full one up to
one float32 rounding; the change measure on a hand-worked vector; the reference
is the last step that ran every block (a planted "previous step" reading fails).
"""
import math

import numpy as np

import synth
from oracle import dit, fbcache, rope

TINY = synth.TINY


def _case(seed=21, L=3, h=3, w=3):
    W = synth.Weights(seed=seed, dims=TINY)
    tabs = rope.token_tables(L, h, w, axes=TINY.axes)
    img = synth.input_f32(seed, 0, (h * w, TINY.patch))
    txt = synth.input_f32(seed, 1, (L, TINY.hidden))
    return W, img, txt, tabs


def test_rel_change_worked_example():
    ref = np.array([1.0, -2.0, 3.0, -4.0], np.float32)
    r = np.array([1.5, -2.0, 2.0, -4.0], np.float32)
    # |0.5| + 0 + |-1| + 0 = 1.5 over |1| + |-2| + |3| + |-4| = 10
    assert fbcache.rel_change(r, ref) == 0.15
    assert fbcache.rel_change(ref, ref) == 0.0
    assert fbcache.rel_change(4 * r, 4 * ref) == 0.15          # scale-free
    assert fbcache.rel_change(np.zeros(3), np.zeros(3)) == 0.0
    assert fbcache.rel_change(np.ones(3), np.zeros(3)) == math.inf


def test_threshold_zero_is_the_plain_pass():
    W, img, txt, tabs = _case()
    st = fbcache.FBCacheState()
    for k, t in enumerate((0.9, 0.7, 0.5)):
        x = (img + 0.01 * k).astype(np.float32)
        got, rel, skip = fbcache.dit_forward_fbcache(W, x, txt, t, *tabs, st, 0.0, k == 0)
        assert not skip and (k == 0) == math.isinf(rel)
        assert np.array_equal(got, dit.dit_forward(W, x, txt, t, *tabs))


def test_repeated_input_is_skipped_and_reproduces_the_pass():
    W, img, txt, tabs = _case(seed=22)
    st = fbcache.FBCacheState()
    full, rel0, s0 = fbcache.dit_forward_fbcache(W, img, txt, 0.6, *tabs, st, 1e9, True)
    again, rel1, s1 = fbcache.dit_forward_fbcache(W, img, txt, 0.6, *tabs, st, 1e9, False)
    assert not s0 and s1 and rel1 == 0.0
    # x1 + (x_last - x1) differs from x_last by at most one rounding per element
    assert np.abs(again - full).max() <= 1e-5 * np.abs(full).max()
    # a new prompt always runs every block, even under an infinite threshold
    _, rel2, s2 = fbcache.dit_forward_fbcache(W, img, txt, 0.6, *tabs, st, math.inf, True)
    assert not s2 and math.isinf(rel2)


def test_skip_adds_the_stored_rest_to_block0_output():
    """A skipped pass's velocity is head(x1 + rest) with x1 from this pass's block 0."""
    W, img, txt, tabs = _case(seed=23)
    L = txt.shape[0]
    st = fbcache.FBCacheState()
    fbcache.dit_forward_fbcache(W, img, txt, 0.6, *tabs, st, 1e9, True)
    x2 = (img + 0.05).astype(np.float32)
    got, _, skip = fbcache.dit_forward_fbcache(W, x2, txt, 0.55, *tabs, st, 1e9, False)
    assert skip
    mods = dit.row_mods(dit.modulation(W.glob, 0.55), dit.modulation(W.glob, 0.0), L, L + img.shape[0])
    cos = np.concatenate([tabs[0], tabs[2]])
    sin = np.concatenate([tabs[1], tabs[3]])
    x1 = dit.block_forward(W.block(0), dit.embed(W.glob, x2, txt), mods, L, cos, sin, TINY.heads)
    assert np.array_equal(got, dit.head(W.glob, (x1[L:] + st.rest).astype(np.float32)))


def test_reference_is_the_last_full_step():
    """Residuals drifting 5 % per step: with the 0.08 threshold the reference stays at the
    last full step, so the drift forces a full step every other call. A reading that
    compares with the previous step would skip every call after the first."""
    base = synth.input_f32(24, 0, (16, 8))
    seq = [(base * (1 + 0.05 * k)).astype(np.float32) for k in range(6)]

    def run(decide):
        st = fbcache.FBCacheState()
        out = []
        for k, r0 in enumerate(seq):
            rel, skip = decide(st, r0, 0.08, k == 0)
            if not skip:
                st.r0 = r0
            out.append(skip)
        return out

    assert run(fbcache.decide) == [False, True, False, True, False, True]

    def previous_step(st, r0, thr, new):          # planted mistake
        rel, skip = fbcache.decide(st, r0, thr, new)
        st.r0 = r0
        return rel, skip

    assert run(previous_step) != [False, True, False, True, False, True]
