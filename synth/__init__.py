"""Seeded synthetic inputs and random-init weights for the Qwen-Image-2.1 DiT step.

This module is shared by the oracle, the tests and the bench. It holds shapes,
seeds and random draws only: none of the model's arithmetic lives here.

Draw recipe
-----------
* Tensor ``k`` of a weight set with seed ``s`` is drawn in chunks of 2**22
  elements; chunk ``c`` comes from
  ``numpy.random.Generator(PCG64(SeedSequence([s, k, c]))).standard_normal(float32)``.
  Weights and biases (and the ZeroCenterRMSNorm gain) are that draw times
  float32(0.02) (float32(Dims.wstd) in general), rounded to bfloat16 with round-to-nearest-even. They are kept as
  the raw bf16 bit patterns (``uint16``).
* Inputs use stream ids ``1_000_000 + j`` and are plain N(0, 1) float32.
* Global tensors use stream ids 0..12; block ``b`` tensor ``j`` uses
  ``100 + 10*b + j``.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

CHUNK = 1 << 22
WEIGHT_STD = np.float32(0.02)
INPUT_STREAM = 1_000_000


@dataclass(frozen=True)
class Dims:
    """Layer widths of the single-stream DiT (Qwen-Image-2.1 architecture table)."""

    hidden: int = 4096
    heads: int = 32
    head_dim: int = 128
    ffn: int = 12288
    patch: int = 64          # latent channels per image token
    tdim: int = 256          # sinusoidal timestep width
    blocks: int = 32
    axes: tuple = (16, 56, 56)  # RoPE widths per axis (frame, height, width)
    wstd: float = 0.02          # weight draw scale; std * sqrt(hidden) ~ 1.3 at full width

    @property
    def mod(self) -> int:
        return 4 * self.hidden


FULL = Dims()
# Tiny width for brute-force checks. Its weight scale keeps std * sqrt(hidden)
# near the full model's value so attention and the branches matter as much.
TINY = Dims(hidden=64, heads=2, head_dim=32, ffn=192, patch=8, tdim=16, blocks=2,
            axes=(8, 12, 12), wstd=0.16)


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def normal_f32(seed: int, stream: int, n: int, scale=None) -> np.ndarray:
    """N(0,1) float32 draws for one tensor, chunked so that chunks draw in parallel."""
    out = np.empty(n, np.float32)
    nchunks = (n + CHUNK - 1) // CHUNK

    def work(c):
        lo = c * CHUNK
        hi = min(n, lo + CHUNK)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, c])))
        g.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])
        if scale is not None:
            out[lo:hi] *= scale

    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(min(_threads(), nchunks)) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.float32).reshape(-1)
    u = a.view(np.uint32)
    out = np.empty(a.size, np.uint16)
    n = a.size

    def work(c):
        lo = c * CHUNK
        hi = min(n, lo + CHUNK)
        x = u[lo:hi]
        r = (x >> np.uint32(16)) & np.uint32(1)
        r += np.uint32(0x7FFF)
        r += x
        r >>= np.uint32(16)
        out[lo:hi] = r

    nchunks = (n + CHUNK - 1) // CHUNK
    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(min(_threads(), nchunks)) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def weight_bf16(seed: int, stream: int, shape, std=WEIGHT_STD) -> np.ndarray:
    n = int(np.prod(shape))
    return f32_to_bf16_bits(normal_f32(seed, stream, n, np.float32(std))).reshape(shape)


# ----------------------------------------------------------------------------- weights

GLOBAL_TENSORS = (
    # name, shape(d), stream id
    ("t_w1", lambda d: (d.hidden, d.tdim), 0),
    ("t_b1", lambda d: (d.hidden,), 1),
    ("t_w2", lambda d: (d.hidden, d.hidden), 2),
    ("t_b2", lambda d: (d.hidden,), 3),
    ("mod_w", lambda d: (d.mod, d.hidden), 4),
    ("mod_b", lambda d: (d.mod,), 5),
    ("txt_norm_w", lambda d: (d.hidden,), 6),
    ("txt_w", lambda d: (d.hidden, d.hidden), 7),
    ("txt_b", lambda d: (d.hidden,), 8),
    ("img_w", lambda d: (d.hidden, d.patch), 9),
    ("img_b", lambda d: (d.hidden,), 10),
    ("out_w", lambda d: (d.patch, d.hidden), 11),
    ("out_b", lambda d: (d.patch,), 12),
)

BLOCK_TENSORS = (
    ("wq", lambda d: (d.hidden, d.hidden), 0),
    ("wk", lambda d: (d.hidden, d.hidden), 1),
    ("wv", lambda d: (d.hidden, d.hidden), 2),
    ("wo", lambda d: (d.hidden, d.hidden), 3),
    ("wg", lambda d: (d.ffn, d.hidden), 4),
    ("wu", lambda d: (d.ffn, d.hidden), 5),
    ("wd", lambda d: (d.hidden, d.ffn), 6),
)


def block_stream(b: int, j: int) -> int:
    return 100 + 10 * b + j


def global_weights(seed: int, dims: Dims = FULL) -> dict:
    """Global tensors (timestep MLP, shared modulation, text/image projections, head)."""
    return {name: weight_bf16(seed, k, shp(dims), dims.wstd) for name, shp, k in GLOBAL_TENSORS}


def block_weights(seed: int, b: int, dims: Dims = FULL) -> dict:
    """The seven bf16 matrices of block ``b``: [out, in] row-major."""
    return {name: weight_bf16(seed, block_stream(b, j), shp(dims), dims.wstd)
            for name, shp, j in BLOCK_TENSORS}


@dataclass
class Weights:
    """A full weight set: global tensors plus a lazily drawn, cached list of blocks."""

    seed: int
    dims: Dims = FULL
    nblocks: int = None
    glob: dict = None
    _blocks: dict = field(default_factory=dict)

    def __post_init__(self):
        if self.nblocks is None:
            self.nblocks = self.dims.blocks
        if self.glob is None:
            self.glob = global_weights(self.seed, self.dims)

    def block(self, b: int) -> dict:
        if b not in self._blocks:
            self._blocks[b] = block_weights(self.seed, b, self.dims)
        return self._blocks[b]


# ----------------------------------------------------------------------------- inputs


def input_f32(seed: int, j: int, shape) -> np.ndarray:
    """N(0,1) float32 input tensor from stream 1_000_000 + j."""
    return normal_f32(seed, INPUT_STREAM + j, int(np.prod(shape))).reshape(shape)


@dataclass(frozen=True)
class StepCase:
    """One DiT call's shapes: L text rows and an h x w image grid."""

    name: str
    seed: int
    L: int
    h: int
    w: int
    timestep: float

    @property
    def N(self) -> int:
        return self.h * self.w


# The five workloads. Sizes follow the host contract: one token per 16x16 px tile.
BLOCK_CASE = StepCase("one block, 128^2, L=8", 0, 8, 8, 8, 0.5)
STEP_256 = StepCase("32 blocks, 256^2, L=22", 1, 22, 16, 16, 0.97)
STEP_384_L22 = StepCase("32 blocks, 384^2, L=22", 2, 22, 24, 24, None)
STEP_384_L494 = StepCase("32 blocks, 384^2, L=494", 2, 494, 24, 24, None)
LOOP_1024 = StepCase("40-step loop, 1024^2, L=407", 3, 407, 64, 64, None)
STEP_2048 = StepCase("32 blocks, 2048^2, L=512", 4, 512, 128, 128, None)

# input stream ids
J_IMG = 0        # img_tokens [N, 64] (or block hidden [L+N, hidden])
J_TXT = 1        # txt_feats [L, hidden]
J_NOISE = 2      # initial latent z [64, h, w] (channel-major)
J_TXT_LONG = 3   # the second prompt of the 384^2 case


def img_tokens(case: StepCase, dims: Dims = FULL) -> np.ndarray:
    return input_f32(case.seed, J_IMG, (case.N, dims.patch))


def txt_feats(case: StepCase, dims: Dims = FULL, j: int = J_TXT) -> np.ndarray:
    return input_f32(case.seed, j, (case.L, dims.hidden))


def block_hidden(case: StepCase, dims: Dims = FULL) -> np.ndarray:
    return input_f32(case.seed, J_IMG, (case.L + case.N, dims.hidden))


def noise_latent(case: StepCase, dims: Dims = FULL) -> np.ndarray:
    """Channel-major initial latent z[c, y, x]."""
    return input_f32(case.seed, J_NOISE, (dims.patch, case.h, case.w))
