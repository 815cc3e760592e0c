"""A small DiT case for profiler captures (same kernels and shapes per launch as 1024^2).

    python -m diffusion_transformer_text_gb300.profile_case [--blocks 2] [--steps 2] [--N 4096] [--L 407] [--mxfp8]

Builds a handle with `blocks` blocks of random-init bf16 weights drawn on the
device, packs a noise latent, runs one joint step (text K/V capture) and then
`steps` image-only steps at N image tokens and L text rows, each followed by the
Euler update, and prints the wall time. With two
blocks it holds about 1.5 GB on the device (weights alone exceed the L2), so a
full profiler capture of one launch stays small. Launch order per pass: text
GEMM (joint only), then per block QKV GEMM, attention, out-projection GEMM,
gate/up GEMM, down GEMM. With --mxfp8 the block GEMMs run on MXFP8 operands
(an activation quantiser launch before each of them).
"""
from __future__ import annotations

import argparse
import time

import numpy as np


def main():
    import torch

    import diffusion_transformer_text_gb300 as qi
    import synth

    ap = argparse.ArgumentParser()
    ap.add_argument("--blocks", type=int, default=2)
    ap.add_argument("--steps", type=int, default=2)
    ap.add_argument("--N", type=int, default=4096)
    ap.add_argument("--L", type=int, default=407)
    ap.add_argument("--mxfp8", action="store_true")
    a = ap.parse_args()
    h = w = int(round(a.N ** 0.5))
    assert h * w == a.N, "N must be a square grid"
    qi.build()
    dev = torch.device("cuda", 0)
    d = qi.DiT(blocks=a.blocks, L_max=a.L, N_max=a.N, mxfp8=a.mxfp8)
    g = torch.Generator(device=dev)
    g.manual_seed(7)

    def t(*shape):
        return (torch.randn(*shape, generator=g, device=dev) * 0.02).to(torch.bfloat16)

    dims = synth.FULL
    d.load_global({n: t(*s(dims)) for n, s, _ in synth.GLOBAL_TENSORS})
    for b in range(a.blocks):
        d.load_block(b, {n: t(*s(dims)) for n, s, _ in synth.BLOCK_TENSORS})
    d.set_mxfp8(a.mxfp8)
    tc, ts, ic, is_ = qi.rope_tables(a.L, h, w)
    txt = torch.randn(a.L, 4096, generator=g, device=dev)
    x = qi.pack_noise(torch.randn(64, h, w, generator=g, device=dev))
    sig, tsteps = qi.flow_sigmas(40, a.N)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    vel = d.step(x, txt, float(np.float32(tsteps[0]) / np.float32(1000)), tc, ts, ic, is_)
    qi.euler_update(x, vel, float(sig[0]), float(sig[1]))
    for i in range(1, a.steps + 1):
        vel = d.step_cached(x, a.L, float(np.float32(tsteps[i]) / np.float32(1000)), ic, is_, vel=vel)
        qi.euler_update(x, vel, float(sig[i]), float(sig[i + 1]))
    torch.cuda.synchronize()
    d.check()
    print(f"profile case: blocks {a.blocks}, N {a.N}, L {a.L}, mxfp8 {a.mxfp8}, 1 joint + {a.steps} image-only steps, "
          f"{(time.perf_counter() - t0) * 1e3:.1f} ms")
    d.close()


if __name__ == "__main__":
    main()
