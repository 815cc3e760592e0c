"""Pins for oracle/dit.py: brute-force loops on a tiny width, invariants, sizes the pages print."""
import math
import os

import numpy as np

import synth
from oracle import dit, rope

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "model_pins.txt")
TINY = synth.TINY


def _golden():
    out = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, *v = line.split()
                out[k] = [float(x) for x in v]
    return out


def _tables(L, h, w, dims):
    return rope.token_tables(L, h, w, axes=dims.axes)


# ---------------------------------------------------------------- loop-form pieces


def _loop_linear(x, w_bits, b_bits=None):
    W = synth.bf16_bits_to_f32(w_bits).astype(np.float64)
    B = None if b_bits is None else synth.bf16_bits_to_f32(b_bits).astype(np.float64)
    out = []
    for o in range(W.shape[0]):
        acc = math.fsum(float(W[o, i]) * float(x[i]) for i in range(W.shape[1]))
        out.append(acc + (0.0 if B is None else float(B[o])))
    return out


def _loop_silu(v):
    return [a / (1.0 + math.exp(-a)) for a in v]


def _loop_modulation(g, t, tdim):
    half = tdim // 2
    s = 1000.0 * t
    e = [math.cos(s * 10000.0 ** (-k / half)) for k in range(half)]
    e += [math.sin(s * 10000.0 ** (-k / half)) for k in range(half)]
    h1 = _loop_silu(_loop_linear(e, g["t_w1"], g["t_b1"]))
    temb = _loop_linear(h1, g["t_w2"], g["t_b2"])
    return _loop_linear(_loop_silu(temb), g["mod_w"], g["mod_b"])


def _loop_norm(row):
    ms = math.fsum(a * a for a in row) / len(row)
    return [a / math.sqrt(ms + dit.EPS) for a in row]


# ---------------------------------------------------------------- tests


def test_timestep_embedding_at_zero_and_order():
    e = dit.timestep_embedding(0.0, 256)
    assert (e[:128] == 1.0).all() and (e[128:] == 0.0).all()
    e = dit.timestep_embedding(0.001, 256)       # argument 1000 * t = 1 at omega_0 = 1
    assert abs(e[0] - math.cos(1.0)) < 1e-6 and abs(e[128] - math.sin(1.0)) < 1e-6
    # last frequency is 10000^(-127/128)
    assert abs(e[127] - math.cos(10000.0 ** (-127 / 128))) < 1e-6


def test_modulation_matches_loops():
    W = synth.Weights(seed=11, dims=TINY)
    for t in (0.0, 0.37, 1.0):
        got = dit.modulation(W.glob, t)
        ref = np.array(_loop_modulation(W.glob, t, TINY.tdim))
        assert np.abs(got - ref).max() <= 1e-5 * max(1.0, np.abs(ref).max())


def test_rmsnorm_closed_forms():
    x = np.full((1, 64), -3.0, np.float32)
    y = dit.rmsnorm(x)
    assert np.allclose(y, -1.0 / math.sqrt(1.0 + dit.EPS / 9.0), rtol=1e-7)
    w = np.full(64, 0.5, np.float32)
    assert np.allclose(dit.zero_center_rmsnorm(x, w), 1.5 * y, rtol=1e-7)


def test_rope_rotation_properties():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 2, 16)).astype(np.float32)
    ang = rng.uniform(-3, 3, (5, 8))
    c, s = np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)
    y = dit.rope(x, c, s)
    # pairwise norms are preserved
    assert np.allclose(np.hypot(y[..., 0::2], y[..., 1::2]), np.hypot(x[..., 0::2], x[..., 1::2]), rtol=1e-5)
    # angle zero is the identity, and the inverse rotation undoes it
    assert np.array_equal(dit.rope(x, np.ones_like(c), np.zeros_like(s)), x)
    assert np.allclose(dit.rope(y, c, -s), x, atol=1e-5)
    # pair j is columns (2j, 2j+1): a pure quarter turn maps (a, b) -> (-b, a)
    q = dit.rope(x, np.zeros_like(c), np.ones_like(s))
    assert np.array_equal(q[..., 0::2], -x[..., 1::2]) and np.array_equal(q[..., 1::2], x[..., 0::2])


def test_block_matches_rowloop():
    W = synth.Weights(seed=5, dims=TINY)
    L, h, w = 3, 2, 2
    R = L + h * w
    tc, ts, ic, is_ = _tables(L, h, w, TINY)
    cos = np.concatenate([tc, ic])
    sin = np.concatenate([ts, is_])
    mods = dit.row_mods(dit.modulation(W.glob, 0.37), dit.modulation(W.glob, 0.0), L, R)
    x = synth.input_f32(5, 0, (R, TINY.hidden))
    got = dit.block_forward(W.block(0), x, mods, L, cos, sin, TINY.heads)
    ref = dit.block_forward_rowloop(W.block(0), x, mods, L, cos, sin, TINY.heads)
    # compare the block's update (output minus input), not the residual-dominated output
    assert np.abs(got - ref).max() <= 2e-5 * np.abs(ref - x).max()


def test_block_rows_equal_dense_block():
    """The selected-rows block (used for full-size sampled checks) equals the dense block."""
    W = synth.Weights(seed=6, dims=TINY)
    L, h, w = 4, 3, 3
    R = L + h * w
    tc, ts, ic, is_ = _tables(L, h, w, TINY)
    cos, sin = np.concatenate([tc, ic]), np.concatenate([ts, is_])
    mods = dit.row_mods(dit.modulation(W.glob, 0.7), dit.modulation(W.glob, 0.0), L, R)
    x = synth.input_f32(6, 0, (R, TINY.hidden))
    dense = dit.block_forward(W.block(0), x, mods, L, cos, sin, TINY.heads)
    rows = [0, 2, 4, 9, 12]
    got, _ = dit.block_forward_rows(W.block(0), x, mods, L, cos, sin, TINY.heads, rows)
    assert np.abs(got - dense[rows]).max() <= 1e-6 * np.abs(dense).max()


def test_dit_matches_loops():
    """Embedding, two blocks and the head, against loop forms (tiny width)."""
    W = synth.Weights(seed=7, dims=TINY)
    L, h, w = 3, 2, 3
    N = h * w
    t = 0.61
    tc, ts, ic, is_ = _tables(L, h, w, TINY)
    img = synth.input_f32(7, 0, (N, TINY.patch))
    txt = synth.input_f32(7, 1, (L, TINY.hidden))
    got = dit.dit_forward(W, img, txt, t, tc, ts, ic, is_)

    g = W.glob
    gain = synth.bf16_bits_to_f32(g["txt_norm_w"]).astype(np.float64)
    rows = []
    for i in range(L):
        nrm = [a * (1.0 + wg) for a, wg in zip(_loop_norm([float(v) for v in txt[i]]), gain)]
        rows.append(_loop_linear(nrm, g["txt_w"], g["txt_b"]))
    for i in range(N):
        rows.append(_loop_linear([float(v) for v in img[i]], g["img_w"], g["img_b"]))
    x = np.array(rows)
    mods = dit.row_mods(np.array(_loop_modulation(g, t, TINY.tdim)),
                        np.array(_loop_modulation(g, 0.0, TINY.tdim)), L, L + N)
    cos = np.concatenate([tc, ic])
    sin = np.concatenate([ts, is_])
    for b in range(TINY.blocks):
        x = dit.block_forward_rowloop(W.block(b), x, mods, L, cos, sin, TINY.heads)
    ref = np.array([_loop_linear(_loop_norm(list(x[L + i])), g["out_w"], g["out_b"]) for i in range(N)])
    assert got.shape == (N, TINY.patch)
    assert np.abs(got - ref).max() <= 5e-5 * np.abs(ref).max()


def test_text_rows_invariant_to_image_and_t():
    """Text K/V of every block do not depend on the image rows or on t (exact)."""
    W = synth.Weights(seed=8, dims=TINY)
    L, h, w = 4, 3, 3
    tc, ts, ic, is_ = _tables(L, h, w, TINY)
    txt = synth.input_f32(8, 1, (L, TINY.hidden))
    k1, k2 = {}, {}
    v1 = dit.dit_forward(W, synth.input_f32(8, 0, (h * w, TINY.patch)), txt, 0.9, tc, ts, ic, is_, keep=k1)
    v2 = dit.dit_forward(W, synth.input_f32(8, 5, (h * w, TINY.patch)), txt, 0.2, tc, ts, ic, is_, keep=k2)
    assert not np.array_equal(v1, v2)
    for (ka, va), (kb, vb) in zip(k1["kv"], k2["kv"]):
        assert np.array_equal(ka, kb) and np.array_equal(va, vb)
    assert np.array_equal(k1["x_out"][:L], k2["x_out"][:L])


def test_sizes_the_pages_print():
    pins = _golden()
    d = synth.FULL
    # 598 rows (576 image + 22 text) through 32 blocks: about 8.5 TFLOP
    fl = dit.step_flops(R=598, N=576, L=22, joint=True)
    want, tol = pins["flops_598"]
    assert abs(fl / 1e12 - want) <= tol
    # 14.2 GB of bf16 parameters
    n_glob = sum(int(np.prod(shp(d))) for _, shp, _ in synth.GLOBAL_TENSORS)
    n_blk = sum(int(np.prod(shp(d))) for _, shp, _ in synth.BLOCK_TENSORS)
    assert n_blk == dit.block_params(d.hidden, d.ffn) == 218_103_808
    gb = (n_glob + d.blocks * n_blk) * 2 / 1e9
    want, tol = pins["dit_gb"]
    assert abs(gb - want) <= tol
    # text K/V cache: 2 x blocks x tokens x hidden x 2 bytes
    mb = 2 * d.blocks * 494 * d.hidden * 2 / 1e6
    want, tol = pins["kv_cache_mb_494"]
    assert abs(mb - want) <= tol
