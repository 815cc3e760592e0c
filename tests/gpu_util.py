"""Helpers shared by the GPU tests: metrics, the tolerance, weight upload."""
import numpy as np

import synth

# Floating-point bar for bf16-GEMM / fp32-accumulate compute against the fp32
# oracle: per-row cosine >= 0.999 and max|diff| / max|ref| <= 2e-2.
COS_MIN = 0.999
REL_MAX = 2e-2


def row_cos(a, b):
    a = np.asarray(a, np.float64).reshape(a.shape[0], -1)
    b = np.asarray(b, np.float64).reshape(b.shape[0], -1)
    num = (a * b).sum(1)
    den = np.sqrt((a * a).sum(1) * (b * b).sum(1)) + 1e-300
    return num / den


def rel_max(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.abs(got - ref).max() / np.abs(ref).max())


def assert_close(got, ref, what, cos_min=COS_MIN, rel=REL_MAX):
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    c = row_cos(got, ref)
    r = rel_max(got, ref)
    assert c.min() >= cos_min and r <= rel, f"{what}: min row cos {c.min():.6f}, max rel {r:.3e}"
    return c.min(), r


def load_weights(dit, W: "synth.Weights"):
    dit.load_global(W.glob)
    for b in range(dit.blocks):
        dit.load_block(b, W.block(b))


def bf16_tensor(bits, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device)


def f32_tensor(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def f16_tensor(a, device="cuda"):
    """float32 values -> fp16 device tensor (int16 view of the fp16 bits)."""
    import torch
    h = np.ascontiguousarray(np.asarray(a, np.float32).astype(np.float16))
    return torch.from_numpy(h.view(np.int16)).to(device)


def f16_bits_to_f32(bits):
    return np.ascontiguousarray(bits).view(np.float16).astype(np.float32)


FP16_MAX = 65504.0


def check_ranges(dit_ranges, what):
    """The largest |value| of every fp16 operand per block (qi_dit_set_range_probe) must be
    finite and within fp16's range; the margins are written to $QI_RANGE_OUT (JSON lines)
    when that variable is set. Returns the per-kind maxima over blocks."""
    import json
    import os

    import diffusion_transformer_text_gb300 as qi
    r = np.asarray(dit_ranges, np.float64)
    assert np.isfinite(r).all() and (r < FP16_MAX).all(), f"{what}: fp16 operand range exceeded: {r.max(0)}"
    per_kind = {k: float(r[:, i].max()) for i, k in enumerate(qi.RANGE_KINDS)}
    path = os.environ.get("QI_RANGE_OUT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": what, "max_abs": per_kind,
                                "margin_to_65504": {k: FP16_MAX / v if v > 0 else None for k, v in per_kind.items()}})
                    + "\n")
    return per_kind


def range_buffer(dit):
    import torch
    import diffusion_transformer_text_gb300 as qi
    return torch.zeros(dit.blocks, len(qi.RANGE_KINDS), dtype=torch.float32, device="cuda")
