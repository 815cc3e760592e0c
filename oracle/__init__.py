"""Plain, slow, CPU reference (the oracle) for the Qwen-Image-2.1 DiT step.

This package is TEST INFRASTRUCTURE. Only tests/, `__graft_entry__.smoke()` and
the CPU-baseline leg of bench.py may import it. The CUDA path never calls it,
and it shares no code with the CUDA path: the only common module is `synth`,
which draws seeded inputs and weights and holds none of the model's arithmetic.

Modules
-------
rope       3-axis RoPE tables, token positions, noise packing (host contract s4-5)
sched      FlowMatch Euler sigmas, timesteps, Euler update (host contract s6),
           guidance combine and the DPM++ 2M step (MLX page, optional modes)
attention  block-causal attention: masked dense, two-segment, brute force
dit        timestep embedding, shared modulation, block, full DiT, output head
fbcache    first-block cache ("Fast mode") around the DiT pass (MLX page)
mx         MXFP8 block-scaled operands and the block with MXFP8 GEMMs

Everything is numpy float32 (bf16 weights widened exactly); the brute-force
checkers use Python float64 loops on tiny shapes.

Pins: every function here is pinned in tests/test_oracle_*.py against values the
pages print (tests/golden/), closed forms, invariants or brute force.
"""
