"""Pins for oracle/attention.py: brute force, the two-segment decomposition, mask shape."""
import numpy as np

from oracle import attention as att


def _qkv(R, H, D, seed=0, scale=1.0):
    rng = np.random.default_rng(seed)
    return [(rng.standard_normal((R, H, D)) * scale).astype(np.float32) for _ in range(3)]


def test_mask_definition():
    m = att.block_causal_mask(3, 4)
    assert m.shape == (7, 7)
    # text rows: lower triangle over text only
    assert m[0].tolist() == [True] + [False] * 6
    assert m[2].tolist() == [True, True, True] + [False] * 4
    # image rows see every row
    assert m[3:].all()


def test_masked_equals_bruteforce():
    L, N, H, D = 3, 4, 2, 8
    q, k, v = _qkv(L + N, H, D, seed=1)
    ref = att.attention_bruteforce(q, k, v, L)
    got = att.attention_masked(q, k, v, L)
    assert np.abs(got - ref).max() <= 1e-5 * np.abs(ref).max()


def test_two_segment_equals_masked():
    L, N, H, D = 9, 23, 3, 16
    q, k, v = _qkv(L + N, H, D, seed=2, scale=2.0)
    a = att.attention_masked(q, k, v, L)
    b = att.attention_two_segment(q, k, v, L)
    assert np.abs(a - b).max() <= 1e-6 * np.abs(a).max()


def test_query_chunking_is_exact():
    L, N, H, D = 5, 40, 2, 8
    q, k, v = _qkv(L + N, H, D, seed=3)
    a = att.attention_masked(q, k, v, L, q_chunk=7)
    b = att.attention_masked(q, k, v, L, q_chunk=4096)
    assert np.array_equal(a, b)


def test_text_rows_ignore_image_rows():
    """Changing image q/k/v leaves every text output bit-identical."""
    L, N, H, D = 6, 10, 2, 8
    q, k, v = _qkv(L + N, H, D, seed=4)
    a = att.attention_masked(q, k, v, L)
    q2, k2, v2 = (x.copy() for x in (q, k, v))
    rng = np.random.default_rng(9)
    for x in (q2, k2, v2):
        x[L:] = rng.standard_normal(x[L:].shape).astype(np.float32)
    b = att.attention_masked(q2, k2, v2, L)
    assert np.array_equal(a[:L], b[:L])
    assert not np.array_equal(a[L:], b[L:])


def test_selected_rows_equal_dense():
    L, N, H, D = 6, 30, 2, 8
    q, k, v = _qkv(L + N, H, D, seed=7)
    dense = att.attention_masked(q, k, v, L)
    rows = np.array([0, 3, 5, 6, 17, 35])
    got = att.attention_rows(q[rows], rows, k, v, L)
    assert np.abs(got - dense[rows]).max() <= 1e-6 * np.abs(dense).max()


def test_first_text_row_copies_its_value():
    """Text row 0 sees only key 0, so its output is v[0] exactly."""
    L, N, H, D = 4, 5, 2, 8
    q, k, v = _qkv(L + N, H, D, seed=5)
    out = att.attention_masked(q, k, v, L).reshape(L + N, H, D)
    assert np.allclose(out[0], v[0], rtol=0, atol=1e-7)


def test_uniform_scores_average_values():
    """Identical keys give uniform weights: an image row returns the mean of all v."""
    L, N, H, D = 3, 5, 1, 4
    q, _, v = _qkv(L + N, H, D, seed=6)
    k = np.ones((L + N, H, D), np.float32)
    out = att.attention_masked(q, k, v, L).reshape(L + N, H, D)
    assert np.allclose(out[L + 2], v.mean(axis=0), atol=1e-6)
    assert np.allclose(out[1], v[:2].mean(axis=0), atol=1e-6)
