"""Oracle: MXFP8 block-scaled operands for the DiT's block GEMMs.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Sources: the MLX page ships 4-bit quantised weights and reports an int8
"per_block 32" experiment; the Core AI page names int8 / 4-bit weight
quantisation. The block-scaled variant here is the OCP Microscaling (MX) v1.0
format MXFP8: blocks of 32 consecutive values along the contraction axis share
one scale X = 2^e stored as an unbiased-by-127 byte (E8M0), and each value is
stored as FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
infinities, S.1111.111 is NaN, largest finite 448).

Readings:
* the shared exponent follows the MX definition e = floor(log2(max |v|)) - 8
  (8 = the exponent of E4M3's largest normal), clamped to [-127, 127]; an
  all-zero block takes e = -127;
* v / X is rounded to E4M3 to nearest, ties to even, and magnitudes above 448
  clamp to 448 (the block's largest value can land in [448, 512));
* the four block GEMMs (QKV, out-projection, gate/up, down) take MXFP8 weights
  and MXFP8 activations; the pre-norm GEMMs quantise x * (1 + s) and apply the
  row's 1/rms to the product (a per-row factor commutes with the sum, not with
  the quantiser, so this fixes which tensor is quantised); the text projection,
  image projection, modulation, timestep MLP, head and attention stay float32.
"""
from __future__ import annotations

import math

import numpy as np

from . import dit
from .attention import attention_masked

BLOCK = 32
E4M3_MAX = 448.0
E4M3_EMAX = 8          # exponent of the largest normal, 448 = 1.75 * 2^8
E4M3_EMIN = -6         # smallest normal 2^-6; subnormals are multiples of 2^-9


def e4m3_decode(code: int) -> float:
    """Value of one E4M3 byte (NaN for S.1111.111)."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return s * m * 2.0 ** -9
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([e4m3_decode(c) for c in range(256)], np.float64)


def e4m3_round(q: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest E4M3 value (ties to even), clamping at +-448."""
    q = np.asarray(q, np.float64)
    a = np.abs(q)
    _, E = np.frexp(a)                           # a = f * 2^E, f in [0.5, 1): floor(log2 a) = E - 1
    shift = np.maximum(E - 1, E4M3_EMIN) - 3     # log2 of the E4M3 spacing at a
    r = np.ldexp(np.round(np.ldexp(a, -shift)), shift)   # exact scalings; round() is half-to-even
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, q)


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """Byte codes of values that are exactly E4M3 (as produced by e4m3_round); rounding
    keeps the sign, so a negative value that rounds to zero is -0 (0x80)."""
    v = np.asarray(v, np.float64)
    finite = E4M3_TABLE.copy()
    finite[np.isnan(finite)] = np.inf
    order = np.argsort(finite[:128], kind="stable")            # non-negative codes 0..126
    vals = finite[:128][order]
    idx = np.searchsorted(vals, np.abs(v))
    idx = np.minimum(idx, 126)
    code = order[idx].astype(np.uint8)
    assert np.array_equal(E4M3_TABLE[code], np.abs(v)), "value is not an E4M3 number"
    return np.where(np.signbit(v), code | 0x80, code).astype(np.uint8)   # -0 keeps its sign: 0x80


def shared_exponent(block_amax: np.ndarray) -> np.ndarray:
    """e = floor(log2(amax)) - 8, clamped to [-127, 127]; -127 for an all-zero block."""
    a = np.asarray(block_amax, np.float64)
    _, E = np.frexp(a)                           # a = f * 2^E, f in [0.5, 1)
    e = (E - 1) - E4M3_EMAX
    e = np.where(a > 0, e, -127)
    return np.clip(e, -127, 127).astype(np.int64)


def quantize(v: np.ndarray):
    """MXFP8 along the last axis (a multiple of 32): (E4M3 values as float64, scale
    exponents e [..., n/32]). Value i is elems[i] * 2^e[i // 32]."""
    v = np.asarray(v, np.float64)
    assert v.shape[-1] % BLOCK == 0
    blocks = v.reshape(*v.shape[:-1], v.shape[-1] // BLOCK, BLOCK)
    e = shared_exponent(np.abs(blocks).max(axis=-1))
    q = e4m3_round(blocks * np.exp2(-e)[..., None])
    return q.reshape(v.shape), e


def dequantize(elems: np.ndarray, e: np.ndarray) -> np.ndarray:
    b = elems.reshape(*elems.shape[:-1], elems.shape[-1] // BLOCK, BLOCK)
    return (b * np.exp2(e)[..., None]).reshape(elems.shape)


def fake_quant(v: np.ndarray) -> np.ndarray:
    """Quantise then dequantise (float32; every MXFP8 value is exact in float32)."""
    q, e = quantize(v)
    return dequantize(q, e).astype(np.float32)


def mx_linear(a: np.ndarray, w_bits) -> np.ndarray:
    """a . W^T with both operands in MXFP8 along the contraction axis (float32 result)."""
    return (fake_quant(a) @ fake_quant(dit.f32(w_bits)).T).astype(np.float32)


def _rinv(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, np.float32)
    ms = np.mean(x * x, axis=-1, keepdims=True, dtype=np.float32)
    return (np.float32(1.0) / np.sqrt(ms + np.float32(dit.EPS))).astype(np.float32)


def block_forward(bw: dict, x: np.ndarray, mods: np.ndarray, L: int, cos, sin, heads: int,
                  return_kv: bool = False):
    """The single-stream block with its four GEMMs in MXFP8 (readings above)."""
    R, H = x.shape
    D = H // heads
    s1, g1, s2, g2 = dit.mod_chunks(mods)
    xm = (x * (np.float32(1.0) + s1)).astype(np.float32)
    r1 = _rinv(x)
    q = (r1 * mx_linear(xm, bw["wq"])).astype(np.float32).reshape(R, heads, D)
    k = (r1 * mx_linear(xm, bw["wk"])).astype(np.float32).reshape(R, heads, D)
    v = (r1 * mx_linear(xm, bw["wv"])).astype(np.float32).reshape(R, heads, D)
    q, k = dit.rope(q, cos, sin), dit.rope(k, cos, sin)
    o = attention_masked(q, k, v, L)
    x = (x + g1 * mx_linear(o, bw["wo"])).astype(np.float32)
    xm2 = (x * (np.float32(1.0) + s2)).astype(np.float32)
    r2 = _rinv(x)
    gate = (r2 * mx_linear(xm2, bw["wg"])).astype(np.float32)
    up = (r2 * mx_linear(xm2, bw["wu"])).astype(np.float32)
    h = (dit.silu(gate) * up).astype(np.float32)
    y = (x + g2 * mx_linear(h, bw["wd"])).astype(np.float32)
    if return_kv:
        return y, k, v
    return y


def dit_forward(weights, img_tokens, txt_feats, t, txt_cos, txt_sin, img_cos, img_sin, nblocks: int = None):
    """Joint DiT pass with MXFP8 block GEMMs; returns vel [N, patch]."""
    g = weights.glob
    heads = weights.dims.heads
    L = txt_feats.shape[0]
    R = L + img_tokens.shape[0]
    mods = dit.row_mods(dit.modulation(g, t), dit.modulation(g, 0.0), L, R)
    cos = np.concatenate([txt_cos, img_cos], axis=0)
    sin = np.concatenate([txt_sin, img_sin], axis=0)
    x = dit.embed(g, img_tokens, txt_feats)
    nb = weights.nblocks if nblocks is None else nblocks
    for b in range(nb):
        x = block_forward(weights.block(b), x, mods, L, cos, sin, heads)
    return dit.head(g, x[L:])
