"""Oracle: the Qwen-Image-2.1 single-stream DiT forward pass, plain numpy float32.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Sources
-------
* Qwen-Image-2.1 Core AI port page, architecture table, DiT row: 32 single-stream
  blocks, ONE modulation Linear 4096 -> 16384 shared by all blocks with one row
  for the sampled t and one for t = 0, a ZeroCenterRMSNorm text projection,
  a three-matrix SwiGLU, 3-axis interleaved RoPE and block-causal attention.
  Graph I/O: img_tokens [1,N,64], txt_feats [1,L,4096], timestep [1],
  txt/img cos and sin [1,.,64] -> vel [1,N,64].
* MLX page, "Text K/V reuse": text rows use the t = 0 modulation row and attend
  causally over text only; `proj_out` is the output head.
* Host contract section 6: the DiT's timestep input is t = timesteps[i] / 1000.

Readings where the pages leave a step open:
* timestep embedding: 256-wide sinusoid [cos | sin] of 1000*t with
  omega_k = 10000^(-k/128), then Linear 256->4096, SiLU, Linear 4096->4096;
* modulation: mod = Linear(SiLU(temb)) 4096->16384, split in that order into
  (s1, g1, s2, g2); a norm is modulated as norm(x) * (1 + s), gates are plain;
* RMSNorm eps = 1e-6 with no learnable gain inside blocks; ZeroCenterRMSNorm
  gain is (1 + w);
* no q/k norm inside the DiT; attention scale 1/sqrt(128);
* biases on the timestep MLP, modulation, img_in, txt_in and proj_out; none on
  QKV, out-projection or SwiGLU;
* the output head is RMSNorm (no gain, no modulation) then proj_out 4096->64.

All arithmetic is float32 on bf16 weights widened exactly to float32.
"""
from __future__ import annotations

import math

import numpy as np

from synth import bf16_bits_to_f32

from .attention import attention_masked, attention_rows

EPS = 1e-6


def f32(w) -> np.ndarray:
    """bf16 bit pattern -> float32 (exact)."""
    return bf16_bits_to_f32(w)


def silu(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, np.float32)
    return (x / (np.float32(1.0) + np.exp(-x))).astype(np.float32)


def rmsnorm(x: np.ndarray, eps: float = EPS) -> np.ndarray:
    x = np.asarray(x, np.float32)
    ms = np.mean(x * x, axis=-1, keepdims=True, dtype=np.float32)
    return (x / np.sqrt(ms + np.float32(eps))).astype(np.float32)


def zero_center_rmsnorm(x: np.ndarray, w: np.ndarray, eps: float = EPS) -> np.ndarray:
    return (rmsnorm(x, eps) * (np.float32(1.0) + w)).astype(np.float32)


def linear(x, w_bits, b_bits=None) -> np.ndarray:
    y = np.asarray(x, np.float32) @ f32(w_bits).T
    if b_bits is not None:
        y = y + f32(b_bits)
    return y.astype(np.float32)


def timestep_embedding(t, dim: int = 256) -> np.ndarray:
    half = dim // 2
    s = np.float32(1000.0) * np.float32(t)
    k = np.arange(half, dtype=np.float32)
    omega = (np.float32(10000.0) ** (-k / np.float32(half))).astype(np.float32)
    arg = (s * omega).astype(np.float32)
    return np.concatenate([np.cos(arg), np.sin(arg)]).astype(np.float32)


def modulation(g: dict, t) -> np.ndarray:
    """The shared modulation row for timestep t: [4*hidden] float32."""
    e = timestep_embedding(t, g["t_w1"].shape[1])
    temb = linear(silu(linear(e[None, :], g["t_w1"], g["t_b1"])), g["t_w2"], g["t_b2"])
    return linear(silu(temb), g["mod_w"], g["mod_b"])[0]


def mod_chunks(mod_row: np.ndarray):
    """(s1, g1, s2, g2) views of one modulation row."""
    H = mod_row.shape[-1] // 4
    return mod_row[..., 0:H], mod_row[..., H:2 * H], mod_row[..., 2 * H:3 * H], mod_row[..., 3 * H:4 * H]


def rope(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Interleaved rotary: pair j = columns (2j, 2j+1) of every head, angle column j.

    x [R, heads, D]; cos, sin [R, D/2].
    """
    a = x[..., 0::2]
    b = x[..., 1::2]
    c = cos[:, None, :]
    s = sin[:, None, :]
    out = np.empty_like(x)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out.astype(np.float32)


def row_mods(mod_img: np.ndarray, mod_txt: np.ndarray, L: int, R: int) -> np.ndarray:
    """Per-row modulation [R, 4H]: text rows (i < L) take the t = 0 row."""
    rows = np.empty((R, mod_img.shape[0]), np.float32)
    rows[:L] = mod_txt
    rows[L:] = mod_img
    return rows


def block_qkv(bw: dict, x: np.ndarray, s1: np.ndarray, cos, sin, heads: int):
    """Pre-attention norm, QKV projection and RoPE: returns q, k, v [R, heads, D]."""
    R, H = x.shape
    D = H // heads
    xn = (rmsnorm(x) * (np.float32(1.0) + s1)).astype(np.float32)
    q = linear(xn, bw["wq"]).reshape(R, heads, D)
    k = linear(xn, bw["wk"]).reshape(R, heads, D)
    v = linear(xn, bw["wv"]).reshape(R, heads, D)
    return rope(q, cos, sin), rope(k, cos, sin), v


def block_after_attention(bw: dict, x: np.ndarray, o: np.ndarray, g1, s2, g2) -> np.ndarray:
    """Out-projection with gate and residual, then the gated SwiGLU MLP with residual."""
    x = (x + g1 * linear(o, bw["wo"])).astype(np.float32)
    xn2 = (rmsnorm(x) * (np.float32(1.0) + s2)).astype(np.float32)
    h = (silu(linear(xn2, bw["wg"])) * linear(xn2, bw["wu"])).astype(np.float32)
    return (x + g2 * linear(h, bw["wd"])).astype(np.float32)


def block_forward(bw: dict, x: np.ndarray, mods: np.ndarray, L: int, cos, sin, heads: int,
                  return_kv: bool = False):
    """One single-stream block over R = L + N rows (text first). mods is [R, 4H]."""
    s1, g1, s2, g2 = mod_chunks(mods)
    q, k, v = block_qkv(bw, x, s1, cos, sin, heads)
    o = attention_masked(q, k, v, L)
    y = block_after_attention(bw, x, o, g1, s2, g2)
    if return_kv:
        return y, k, v
    return y


def block_forward_rows(bw: dict, x: np.ndarray, mods: np.ndarray, L: int, cos, sin, heads: int, rows,
                       kv=None):
    """The block's output for selected global rows only.

    Every row's K and V are still needed (x, mods, cos, sin cover all R rows);
    pass `kv` = (k, v) [R, heads, D] to reuse them. Returns (out [n, H], (k, v)).
    """
    rows = np.asarray(rows)
    s1, g1, s2, g2 = mod_chunks(mods)
    if kv is None:
        _, k, v = block_qkv(bw, x, s1, cos, sin, heads)
    else:
        k, v = kv
    q, _, _ = block_qkv(bw, x[rows], s1[rows], cos[rows], sin[rows], heads)
    o = attention_rows(q, rows, k, v, L)
    out = block_after_attention(bw, x[rows], o, g1[rows], s2[rows], g2[rows])
    return out, (k, v)


def embed(g: dict, img_tokens, txt_feats):
    """img_in(img_tokens) and txt_in(ZeroCenterRMSNorm(txt_feats)), concatenated text first."""
    txt = linear(zero_center_rmsnorm(txt_feats, f32(g["txt_norm_w"])), g["txt_w"], g["txt_b"])
    img = linear(img_tokens, g["img_w"], g["img_b"])
    return np.concatenate([txt, img], axis=0).astype(np.float32)


def head(g: dict, x_img: np.ndarray) -> np.ndarray:
    """Output head on image rows: RMSNorm then proj_out."""
    return linear(rmsnorm(x_img), g["out_w"], g["out_b"])


def dit_forward(weights, img_tokens, txt_feats, t, txt_cos, txt_sin, img_cos, img_sin,
                nblocks: int = None, keep=None):
    """Full joint DiT pass; returns vel [N, patch].

    weights: synth.Weights. `keep`, if a dict, receives per-block text K/V
    (key "kv") and the residual stream entering every block (key "x").
    """
    g = weights.glob
    heads = weights.dims.heads
    L = txt_feats.shape[0]
    N = img_tokens.shape[0]
    R = L + N
    mods = row_mods(modulation(g, t), modulation(g, 0.0), L, R)
    cos = np.concatenate([txt_cos, img_cos], axis=0)
    sin = np.concatenate([txt_sin, img_sin], axis=0)
    x = embed(g, img_tokens, txt_feats)
    nb = weights.nblocks if nblocks is None else nblocks
    for b in range(nb):
        if keep is not None:
            keep.setdefault("x", []).append(x.copy())
        x, k, v = block_forward(weights.block(b), x, mods, L, cos, sin, heads, return_kv=True)
        if keep is not None:
            keep.setdefault("kv", []).append((k[:L].copy(), v[:L].copy()))
    if keep is not None:
        keep["x_out"] = x.copy()
    return head(g, x[L:])


# ----------------------------------------------------------------------------- brute force


def block_forward_rowloop(bw: dict, x, mods, L: int, cos, sin, heads: int):
    """The same block as `block_forward`, one row and one output at a time in
    Python floats (float64). Written without numpy broadcasting, for tiny widths."""
    R, H = x.shape
    D = H // heads
    W = {k_: f32(v_).astype(np.float64).tolist() for k_, v_ in bw.items()}
    X = np.asarray(x, np.float64).tolist()
    M = np.asarray(mods, np.float64).tolist()
    C = np.asarray(cos, np.float64).tolist()
    S = np.asarray(sin, np.float64).tolist()

    def norm(row):
        ms = sum(e * e for e in row) / len(row)
        r = 1.0 / math.sqrt(ms + EPS)
        return [e * r for e in row]

    def matvec(mat, vec):
        return [sum(m_ * v_ for m_, v_ in zip(mrow, vec)) for mrow in mat]

    def rotate(vec, r):
        out = list(vec)
        for hh in range(heads):
            for j in range(D // 2):
                a, b = vec[hh * D + 2 * j], vec[hh * D + 2 * j + 1]
                c, s = C[r][j], S[r][j]
                out[hh * D + 2 * j] = a * c - b * s
                out[hh * D + 2 * j + 1] = a * s + b * c
        return out

    qs, ks, vs = [], [], []
    for r in range(R):
        s1 = M[r][0:H]
        xn = [a * (1.0 + s) for a, s in zip(norm(X[r]), s1)]
        qs.append(rotate(matvec(W["wq"], xn), r))
        ks.append(rotate(matvec(W["wk"], xn), r))
        vs.append(matvec(W["wv"], xn))
    out = []
    for r in range(R):
        g1 = M[r][H:2 * H]
        s2 = M[r][2 * H:3 * H]
        g2 = M[r][3 * H:4 * H]
        keys = range(r + 1) if r < L else range(R)
        o = [0.0] * H
        for hh in range(heads):
            sc = [sum(qs[r][hh * D + d] * ks[j][hh * D + d] for d in range(D)) / math.sqrt(D) for j in keys]
            mx = max(sc)
            ws = [math.exp(s - mx) for s in sc]
            tot = sum(ws)
            for d in range(D):
                o[hh * D + d] = sum(w_ * vs[j][hh * D + d] for w_, j in zip(ws, keys)) / tot
        att = matvec(W["wo"], o)
        x1 = [a + g * b for a, g, b in zip(X[r], g1, att)]
        xn2 = [a * (1.0 + s) for a, s in zip(norm(x1), s2)]
        gate = matvec(W["wg"], xn2)
        up = matvec(W["wu"], xn2)
        hid = [(gv / (1.0 + math.exp(-gv))) * uv for gv, uv in zip(gate, up)]
        dn = matvec(W["wd"], hid)
        out.append([a + g * b for a, g, b in zip(x1, g2, dn)])
    return np.array(out, dtype=np.float64)


# ----------------------------------------------------------------------------- accounting


def block_params(hidden: int, ffn: int) -> int:
    """Parameters of one block: Q, K, V, out (hidden^2 each) and three SwiGLU matrices."""
    return 4 * hidden * hidden + 3 * hidden * ffn


def step_flops(R: int, N: int, L: int, joint: bool, hidden=4096, ffn=12288, blocks=32) -> int:
    """Algorithmic FLOPs of one DiT pass (matmuls and attention; elementwise work excluded).

    GEMMs: 2 * R * block_params per block. Attention: each image query scores and
    mixes L + N keys (4 * hidden FLOP per pair); on the joint pass the text queries
    add L(L+1)/2 causal pairs.
    """
    gemm = 2 * R * block_params(hidden, ffn)
    att = N * (N + L) * 4 * hidden
    if joint:
        att += L * (L + 1) // 2 * 4 * hidden
    return blocks * (gemm + att)
