"""Pins for oracle/mx.py: the E4M3 format, the MX shared exponent and rounding, and the
MXFP8 block against the float32 block.

The E4M3 values follow from the format's definition (sign, exponent bias 7, three
mantissa bits, S.1111.111 = NaN); ties-to-even is checked on every adjacent pair;
the block structure reduces to the float32 oracle block when quantisation is the
identity.
"""
import math

import numpy as np
import pytest

import synth
from oracle import dit, mx, rope

TINY = synth.TINY


def test_e4m3_table_closed_forms():
    t = mx.E4M3_TABLE
    assert t[0x38] == 1.0 and t[0x40] == 2.0 and t[0xB8] == -1.0
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0
    assert t[0x01] == 2.0 ** -9 and t[0x08] == 2.0 ** -6 and t[0x07] == 7 * 2.0 ** -9
    assert math.isnan(t[0x7F]) and math.isnan(t[0xFF])
    assert t[0x80] == 0.0 and math.copysign(1.0, t[0x80]) == -1.0
    pos = t[:127]
    assert (np.diff(pos) > 0).all()                      # codes 0..126 increase
    assert np.isfinite(t).sum() == 254


def test_round_is_identity_on_e4m3_and_ties_go_even():
    pos = mx.E4M3_TABLE[:127]
    assert np.array_equal(mx.e4m3_round(pos), pos)
    assert np.array_equal(mx.e4m3_round(-pos), -pos)
    for c in range(126):
        a, b = pos[c], pos[c + 1]
        mid = (a + b) / 2
        even = a if c % 2 == 0 else b                    # the code whose last mantissa bit is 0
        assert mx.e4m3_round(mid) == even, c
        assert mx.e4m3_round(np.nextafter(mid, 0)) == a
        assert mx.e4m3_round(np.nextafter(mid, 1e9)) == b


def test_round_saturates():
    assert mx.e4m3_round(449.0) == 448.0 and mx.e4m3_round(511.9) == 448.0
    assert mx.e4m3_round(1e30) == 448.0 and mx.e4m3_round(-1e30) == -448.0
    assert mx.e4m3_round(2.0 ** -11) == 0.0              # below half the smallest subnormal
    assert mx.e4m3_round(3 * 2.0 ** -11) == 2.0 ** -9    # 0.75 ulp rounds up


def test_shared_exponent():
    e = mx.shared_exponent(np.array([1.0, 448.0, 500.0, 512.0, 2.0 ** -20, 0.0, 1e38, 1e-45]))
    assert e.tolist() == [-8, 0, 0, 1, -28, -127, 118, -127]
    # a block whose largest value lands in [448, 512) clamps that value to 448
    v = np.zeros(32)
    v[3] = 500.0
    q, es = mx.quantize(v[None, :])
    assert es[0, 0] == 0 and q[0, 3] == 448.0


def test_exact_round_trip_and_error_bound():
    rng = np.random.default_rng(3)
    # values that are already E4M3 times 2^k, the block max in [256, 448] * 2^k: exact
    codes = rng.integers(0, 127, size=(64, 32))
    codes[:, 0] = 0x7A                                     # 320, so e = floor(log2 320) - 8 = 0
    vals = mx.E4M3_TABLE[codes] * np.exp2(rng.integers(-20, 20, size=(64, 1)))
    assert np.array_equal(mx.fake_quant(vals).astype(np.float64), vals)
    # random data: every element within half an E4M3 ulp, except a saturated block max
    v = rng.standard_normal((256, 128)) * np.exp2(rng.integers(-10, 10, size=(256, 1)))
    q, e = mx.quantize(v)
    d = mx.dequantize(q, e)
    X = np.repeat(np.exp2(e), 32, axis=-1)
    normal = np.abs(v) >= X * 2.0 ** -6
    sat = np.abs(v / X) > 448
    assert (np.abs(d - v)[normal & ~sat] <= 2.0 ** -4 * np.abs(v)[normal & ~sat]).all()
    assert (np.abs(d - v)[~normal] <= X[~normal] * 2.0 ** -10).all()
    assert (np.abs(d - v)[sat] <= 64 * X[sat]).all()


def test_encode_decodes_back():
    vals = np.array([0.0, 1.0, -2.5, 448.0, -448.0, 2.0 ** -9, -(2.0 ** -6), -0.0])
    codes = mx.e4m3_encode(vals)
    assert np.array_equal(mx.E4M3_TABLE[codes], vals)
    assert codes.tolist() == [0x00, 0x38, 0xC2, 0x7E, 0xFE, 0x01, 0x88, 0x80]
    assert mx.e4m3_encode(mx.e4m3_round(np.array([-1e-5]))).tolist() == [0x80]


def test_mx_linear_is_the_dequantized_product():
    rng = np.random.default_rng(4)
    a = rng.standard_normal((5, 64)).astype(np.float32)
    w = synth.f32_to_bf16_bits(rng.standard_normal((3, 64)).astype(np.float32)).reshape(3, 64)
    qa, ea = mx.quantize(a)
    qw, ew = mx.quantize(dit.f32(w))
    A, W = mx.dequantize(qa, ea), mx.dequantize(qw, ew)
    ref = np.array([[sum(A[i, k] * W[j, k] for k in range(64)) for j in range(3)] for i in range(5)])
    assert np.abs(mx.mx_linear(a, w) - ref).max() <= 1e-6 * np.abs(ref).max()


def test_block_reduces_to_float32_block(monkeypatch):
    """With quantisation switched off the MXFP8 block is the float32 block (the 1/rms is
    applied after the product instead of before: float32 rounding apart)."""
    W = synth.Weights(seed=31, dims=TINY)
    L, h, w = 3, 2, 3
    R = L + h * w
    tc, ts, ic, is_ = rope.token_tables(L, h, w, axes=TINY.axes)
    cos, sin = np.concatenate([tc, ic]), np.concatenate([ts, is_])
    mods = dit.row_mods(dit.modulation(W.glob, 0.4), dit.modulation(W.glob, 0.0), L, R)
    x = synth.input_f32(31, 0, (R, TINY.hidden))
    ref = dit.block_forward(W.block(0), x, mods, L, cos, sin, TINY.heads)
    monkeypatch.setattr(mx, "fake_quant", lambda v: np.asarray(v, np.float32))
    got = mx.block_forward(W.block(0), x, mods, L, cos, sin, TINY.heads)
    assert np.abs(got - ref).max() <= 1e-5 * np.abs(ref).max()


def test_block_quantisation_changes_the_block():
    """With quantisation on, the block moves by the MXFP8 rounding: well above float32
    noise, well below the block's own update."""
    W = synth.Weights(seed=32, dims=TINY)
    L, h, w = 3, 2, 3
    R = L + h * w
    tc, ts, ic, is_ = rope.token_tables(L, h, w, axes=TINY.axes)
    cos, sin = np.concatenate([tc, ic]), np.concatenate([ts, is_])
    mods = dit.row_mods(dit.modulation(W.glob, 0.4), dit.modulation(W.glob, 0.0), L, R)
    x = synth.input_f32(32, 0, (R, TINY.hidden))
    ref = dit.block_forward(W.block(0), x, mods, L, cos, sin, TINY.heads) - x
    got = mx.block_forward(W.block(0), x, mods, L, cos, sin, TINY.heads) - x
    rel = np.abs(got - ref).max() / np.abs(ref).max()
    assert 1e-4 < rel < 0.2


@pytest.mark.parametrize("bad", ["exponent_minus_7", "round_half_up"])
def test_control_planted_quantiser_mistakes(bad, monkeypatch):
    if bad == "exponent_minus_7":
        orig = mx.shared_exponent
        monkeypatch.setattr(mx, "shared_exponent", lambda a: orig(a) + 1)
        codes = np.random.default_rng(5).integers(0, 127, size=(8, 32))
        codes[:, 0] = 0x7A
        vals = mx.E4M3_TABLE[codes]
        assert not np.array_equal(mx.fake_quant(vals).astype(np.float64), vals)
    else:
        monkeypatch.setattr(mx, "e4m3_round", lambda q: np.copysign(
            np.minimum(np.floor(np.abs(q) / np.exp2(np.maximum(np.floor(np.log2(np.maximum(np.abs(q), 1e-300))),
                                                                -6) - 3) + 0.5)
                       * np.exp2(np.maximum(np.floor(np.log2(np.maximum(np.abs(q), 1e-300))), -6) - 3), 448.0), q))
        pos = mx.E4M3_TABLE[:127]
        mids = (pos[:-1] + pos[1:]) / 2
        evens = np.where(np.arange(126) % 2 == 0, pos[:-1], pos[1:])
        assert not np.array_equal(mx.e4m3_round(mids), evens)


# ----------------------------------------------------------------------------- tolerance
# The library quantises the fp16 copies of its GEMM inputs and runs attention on fp16
# Q / K / V. Rounding a value to fp16 moves it by <= 2^-11 relative, which carries about
# 2^-7 of the E4M3 codes one step (2^-3 relative) away from the float32 oracle's code. The
# GPU tests of the MXFP8 mode use the tolerance below; this test shows that those fp16
# roundings alone, emulated here in numpy on the one-block workload, already use most of it.
MX_BLOCK_COS, MX_BLOCK_REL = 0.999, 5e-2


def _f16(a):
    return np.asarray(a, np.float32).astype(np.float16).astype(np.float32)


def _block_fp16_operands(bw, x, mods, L, cos, sin, heads):
    """oracle/mx.block_forward with every quantiser input and Q / K / V rounded to fp16."""
    R, H = x.shape
    D = H // heads
    s1, g1, s2, g2 = dit.mod_chunks(mods)
    xm = _f16(x * (np.float32(1.0) + s1))
    r1 = mx._rinv(x)
    q = _f16((r1 * mx.mx_linear(xm, bw["wq"])).reshape(R, heads, D))
    k = (r1 * mx.mx_linear(xm, bw["wk"])).reshape(R, heads, D)
    v = _f16((r1 * mx.mx_linear(xm, bw["wv"])).reshape(R, heads, D))
    q, k = _f16(dit.rope(q, cos, sin)), _f16(dit.rope(k, cos, sin))
    o = _f16(mx.attention_masked(q, k, v, L))
    x = (x + g1 * mx.mx_linear(o, bw["wo"])).astype(np.float32)
    xm2 = _f16(x * (np.float32(1.0) + s2))
    r2 = mx._rinv(x)
    h = _f16(dit.silu(r2 * mx.mx_linear(xm2, bw["wg"])) * (r2 * mx.mx_linear(xm2, bw["wu"])))
    return (x + g2 * mx.mx_linear(h, bw["wd"])).astype(np.float32)


@pytest.mark.slow
def test_fp16_operand_roundings_fit_the_mxfp8_tolerance():
    case = synth.BLOCK_CASE
    W = synth.Weights(seed=case.seed, nblocks=1)
    x = synth.block_hidden(case)
    tc, ts, ic, is_ = rope.token_tables(case.L, case.h, case.w)
    cos, sin = np.concatenate([tc, ic]), np.concatenate([ts, is_])
    mods = dit.row_mods(dit.modulation(W.glob, case.timestep), dit.modulation(W.glob, 0.0), case.L,
                        case.L + case.N)
    bw = W.block(0)
    ref = mx.block_forward(bw, x, mods, case.L, cos, sin, 32) - x
    emu = _block_fp16_operands(bw, x, mods, case.L, cos, sin, 32) - x
    f32 = dit.block_forward(bw, x, mods, case.L, cos, sin, 32) - x
    row_cos = (emu * ref).sum(1) / np.linalg.norm(emu, axis=1) / np.linalg.norm(ref, axis=1)
    rel = np.abs(emu - ref).max() / np.abs(ref).max()
    assert row_cos.min() >= MX_BLOCK_COS and rel <= MX_BLOCK_REL
    assert rel > 0.3 * MX_BLOCK_REL                        # the roundings use a real share of it
    # and the emulation stays much closer to the MXFP8 block than that is to float32
    assert np.sqrt(((emu - ref) ** 2).mean()) < 0.75 * np.sqrt(((ref - f32) ** 2).mean())


MX_STEP_COS, MX_STEP_REL = 0.99, 1e-1   # two blocks and the output head (256^2 workload)


@pytest.mark.slow
def test_fp16_operand_roundings_fit_the_mxfp8_step_tolerance():
    case = synth.STEP_256
    nb = 2
    W = synth.Weights(seed=case.seed, nblocks=nb)
    img = synth.img_tokens(case)
    txt = synth.txt_feats(case)
    tabs = rope.token_tables(case.L, case.h, case.w)
    t = np.float32(case.timestep)
    ref = mx.dit_forward(W, img, txt, t, *tabs, nblocks=nb)
    g = W.glob
    L = case.L
    mods = dit.row_mods(dit.modulation(g, t), dit.modulation(g, 0.0), L, L + case.N)
    cos = np.concatenate([tabs[0], tabs[2]])
    sin = np.concatenate([tabs[1], tabs[3]])
    x = dit.embed(g, img, txt)
    for b in range(nb):
        x = _block_fp16_operands(W.block(b), x, mods, L, cos, sin, 32)
    emu = dit.head(g, x[L:])
    row_cos = (emu * ref).sum(1) / np.linalg.norm(emu, axis=1) / np.linalg.norm(ref, axis=1)
    rel = np.abs(emu - ref).max() / np.abs(ref).max()
    assert row_cos.min() >= MX_STEP_COS and rel <= MX_STEP_REL
