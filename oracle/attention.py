"""Oracle: block-causal attention of the single-stream DiT.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Source: Qwen-Image-2.1 Core AI port page, architecture table, DiT row: text rows
are causal over text, image rows are bidirectional and see all text; the port
computes it as two SDPA calls (text->text causal, image->all). The MLX page,
"Text K/V reuse", adds that text rows never see the image.

With L text rows first and R = L + N rows in all, query row i may attend to key
row j iff (i < L and j <= i) or (i >= L). Scores are q.k / sqrt(head_dim).

q, k, v are [R, heads, head_dim] float32 here.
"""
from __future__ import annotations

import math

import numpy as np


def block_causal_mask(L: int, N: int) -> np.ndarray:
    R = L + N
    i = np.arange(R)[:, None]
    j = np.arange(R)[None, :]
    return ((i < L) & (j <= i)) | (i >= L)


def _softmax_rows(s: np.ndarray) -> np.ndarray:
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=-1, keepdims=True)


def attention_masked(q, k, v, L: int, q_chunk: int = 2048) -> np.ndarray:
    """Dense masked softmax over all key rows; the plain definition. Returns [R, heads*dim]."""
    R, H, D = q.shape
    scale = np.float32(1.0 / math.sqrt(D))
    out = np.empty((R, H, D), np.float32)
    N = R - L
    for h in range(H):
        kh = k[:, h, :]
        vh = v[:, h, :]
        for lo in range(0, R, q_chunk):
            hi = min(R, lo + q_chunk)
            s = (q[lo:hi, h, :] @ kh.T) * scale
            i = np.arange(lo, hi)[:, None]
            j = np.arange(R)[None, :]
            allowed = ((i < L) & (j <= i)) | (i >= L)
            s = np.where(allowed, s, -np.inf).astype(np.float32)
            out[lo:hi, h, :] = _softmax_rows(s) @ vh
    del N
    return out.reshape(R, H * D)


def sdpa(q, k, v, causal: bool) -> np.ndarray:
    """One scaled-dot-product attention call, [Rq, H, D] x [Rk, H, D]."""
    Rq, H, D = q.shape
    Rk = k.shape[0]
    scale = np.float32(1.0 / math.sqrt(D))
    out = np.empty((Rq, H, D), np.float32)
    for h in range(H):
        s = (q[:, h, :] @ k[:, h, :].T) * scale
        if causal:
            s = np.where(np.arange(Rk)[None, :] <= np.arange(Rq)[:, None], s, -np.inf).astype(np.float32)
        out[:, h, :] = _softmax_rows(s) @ v[:, h, :]
    return out


def attention_two_segment(q, k, v, L: int) -> np.ndarray:
    """The port's decomposition: SDPA(text q, text k/v, causal) and SDPA(image q, all k/v)."""
    R, H, D = q.shape
    txt = sdpa(q[:L], k[:L], v[:L], causal=True)
    img = sdpa(q[L:], k, v, causal=False)
    return np.concatenate([txt, img], axis=0).reshape(R, H * D)


def attention_rows(q_rows, rows, k, v, L: int) -> np.ndarray:
    """The masked softmax for selected query rows only.

    q_rows [n, H, D] are the queries of global rows `rows`; k, v [R, H, D] hold
    every key row. Row i sees keys 0..i if i < L, else all R keys. Returns [n, H*D].
    """
    n, H, D = q_rows.shape
    R = k.shape[0]
    scale = np.float32(1.0 / math.sqrt(D))
    out = np.empty((n, H, D), np.float32)
    j = np.arange(R)
    for h in range(H):
        s = (q_rows[:, h, :] @ k[:, h, :].T) * scale
        i = np.asarray(rows)[:, None]
        allowed = ((i < L) & (j[None, :] <= i)) | (i >= L)
        s = np.where(allowed, s, -np.inf).astype(np.float32)
        out[:, h, :] = _softmax_rows(s) @ v[:, h, :]
    return out.reshape(n, H * D)


def attention_bruteforce(q, k, v, L: int):
    """Triple loop in Python floats (float64); for tiny shapes only."""
    R, H, D = q.shape
    out = [[[0.0] * D for _ in range(H)] for _ in range(R)]
    for i in range(R):
        keys = list(range(i + 1)) if i < L else list(range(R))
        for h in range(H):
            scores = []
            for j in keys:
                dot = 0.0
                for d in range(D):
                    dot += float(q[i, h, d]) * float(k[j, h, d])
                scores.append(dot / math.sqrt(D))
            m = max(scores)
            ws = [math.exp(s - m) for s in scores]
            tot = sum(ws)
            for d in range(D):
                acc = 0.0
                for w_, j in zip(ws, keys):
                    acc += w_ * float(v[j, h, d])
                out[i][h][d] = acc / tot
    return np.array(out, dtype=np.float64).reshape(R, H * D)
