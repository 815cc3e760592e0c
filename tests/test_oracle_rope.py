"""Pins for oracle/rope.py: the pages' worked example, closed forms and invariants."""
import os

import numpy as np
import pytest

from oracle import rope

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rope_pins.txt")


def _golden():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def test_position_worked_example():
    for row in _golden():
        if row[0] != "hpos_range":
            continue
        h, lo, hi = int(row[1]), int(row[2]), int(row[3])
        pos = rope.image_positions(L=5, h=h, w=h)
        assert pos[:, 1].min() == lo and pos[:, 1].max() == hi
        assert pos[:, 2].min() == lo and pos[:, 2].max() == hi
        assert (pos[:, 0] == 5).all()
        # raster order: token y*w + x
        assert tuple(pos[0]) == (5, lo, lo)
        assert tuple(pos[h + 1]) == (5, lo + 1, lo + 1)
        assert tuple(pos[h - 1]) == (5, lo, hi)


def test_text_positions():
    p = rope.text_positions(7)
    assert (p[:, 0] == np.arange(7)).all() and (p[:, 1] == p[:, 0]).all() and (p[:, 2] == p[:, 0]).all()


def test_table_shape():
    g = {r[0]: r[1:] for r in _golden()}
    tabs = rope.axis_tables()
    assert [t[0].shape for t in tabs] == [(int(g["table_rows"][0]), int(c)) for c in g["table_cols"]]


def test_omega_closed_forms():
    for row in _golden():
        if row[0] != "omega":
            continue
        d, k, val = int(row[1]), int(row[2]), float(row[3])
        assert rope.axis_freqs(d)[k] == np.float32(val)
    # k = 0 is exactly 1 for every axis
    for d in (16, 56):
        assert rope.axis_freqs(d)[0] == np.float32(1.0)


def test_position_zero_is_identity():
    for c, s in rope.axis_tables():
        row = 0 - rope.POS_LO
        assert (c[row] == 1.0).all() and (s[row] == 0.0).all()


def test_axes_1_and_2_byte_identical():
    tabs = rope.axis_tables()
    assert tabs[1][0].tobytes() == tabs[2][0].tobytes()
    assert tabs[1][1].tobytes() == tabs[2][1].tobytes()


def test_unit_modulus_and_symmetry():
    for c, s in rope.axis_tables():
        r = c.astype(np.float64) ** 2 + s.astype(np.float64) ** 2
        assert np.abs(r - 1.0).max() <= 2.0 ** -23
        # positions p and -p: rows 1024 + p and 1024 - p (p <= 1024)
        p = np.arange(1, 1025)
        assert (c[1024 + p] == c[1024 - p]).all()
        assert (s[1024 + p] == -s[1024 - p]).all()


def test_values_against_high_precision():
    """Every sampled entry equals fl32 of the exact cos/sin of its float32 angle."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.prec = 120
    rng = np.random.default_rng(0)
    for d, (c, s) in zip((16, 56), rope.axis_tables((16, 56))):
        w = rope.axis_freqs(d)
        for _ in range(300):
            row = int(rng.integers(0, rope.NPOS))
            k = int(rng.integers(0, d // 2))
            pos = row + rope.POS_LO
            # the float32 angle, formed without numpy: exact product rounded once
            ang = float(np.float32(mpmath.mpf(float(np.float32(pos))) * mpmath.mpf(float(w[k]))))
            assert c[row, k] == np.float32(float(mpmath.cos(ang)))
            assert s[row, k] == np.float32(float(mpmath.sin(ang)))
            # omega itself: correctly rounded 10000^(-2k/d)
            assert w[k] == np.float32(float(mpmath.power(10000, mpmath.mpf(-2 * k) / d)))


def test_token_tables_concatenate_axis_rows():
    L, h, w = 5, 4, 6
    tc, ts, ic, is_ = rope.token_tables(L, h, w)
    a0, a1, a2 = rope.axis_tables()
    assert tc.shape == (L, 64) and ic.shape == (h * w, 64)
    for i in range(L):
        assert (tc[i, :8] == a0[0][i + 1024]).all()
        assert (tc[i, 8:36] == a1[0][i + 1024]).all()
        assert (ts[i, 36:] == a2[1][i + 1024]).all()
    # image token (y=3, x=0): (L, 3 - 2, 0 - 3)
    t = 3 * w + 0
    assert (ic[t, :8] == a0[0][L + 1024]).all()
    assert (ic[t, 8:36] == a1[0][1 + 1024]).all()
    assert (is_[t, 36:] == a2[1][-3 + 1024]).all()


def test_pack_noise_is_the_stated_permutation():
    c, h, w = 3, 2, 4
    z = np.arange(c * h * w, dtype=np.float32).reshape(c, h, w)
    x = rope.pack_noise(z)
    assert x.shape == (h * w, c)
    # x[y*w + x, ch] = z[ch, y, x]; equivalently z.reshape(c, h*w).T
    assert x[1 * w + 2, 1] == z[1, 1, 2]
    assert (x == z.reshape(c, h * w).T).all()
