"""qi_gemm_bf16_noalloc: the GEMM for callers that may not allocate device memory.

Callers inside a host that owns all device memory (a fixed-arena inference
server, a plugin barred from the CUDA allocator) cannot create a qi_dit handle,
since creating one allocates. This entry point keeps its scratch (the kernel's
status word) in a static device array instead.

The test calls it through the C ABI, two calls in a row per shape, and checks
each result against the float64 product of the bf16 operands, within the
bound the GEMM tests use, and, bit for bit, against
qi_gemm_bf16 on a handle, which runs the same kernel with the same grid on the
same device. One shape has a ragged row count (M = 1000: full waves, a last
wave of half tiles and a partial row tile). It also checks the status word is
cleared between calls: a call without the synchronising check, then one with
it, must both succeed. It sits in its own file, collected last, and needs
nothing from earlier tests.
"""
import ctypes

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qi():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import diffusion_transformer_text_gb300 as q
    q.build()
    q.lib()
    return q


def _noalloc(qi, A, B, M, N, K, sync_check=1):
    import torch
    D = torch.full((M, N), float("nan"), dtype=torch.float32, device=A.device)
    st = qi.lib().qi_gemm_bf16_noalloc(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, sync_check,
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, qi.lib().qi_last_error().decode()
    return D


@pytest.mark.parametrize("M,N,K,seed", [(200, 512, 256, 31), (300, 768, 4096, 32), (1000, 4096, 1024, 33)])
def test_noalloc_matches_product_and_handle_gemm_twice(qi, M, N, K, seed):
    import torch
    from gpu_util import bf16_tensor
    A_bits = synth.weight_bf16(seed, 0, (M, K), std=1.0)
    B_bits = synth.weight_bf16(seed, 1, (N, K), std=1.0)
    A, B = bf16_tensor(A_bits), bf16_tensor(B_bits)
    a = synth.bf16_bits_to_f32(A_bits).astype(np.float64)
    b = synth.bf16_bits_to_f32(B_bits).astype(np.float64)
    exact = a @ b.T
    bound = 1e-5 * (np.abs(a) @ np.abs(b).T) + 1e-6  # the GEMM tests' bound
    d = qi.DiT(blocks=1, L_max=8, N_max=64)
    try:
        ref = d.gemm(A, B).cpu().numpy()
        d.check()
    finally:
        d.close()
    for call in range(2):
        got = _noalloc(qi, A, B, M, N, K).cpu().numpy()
        assert np.isfinite(got).all(), f"call {call}"
        err = np.abs(got.astype(np.float64) - exact)
        assert (err <= bound).all(), f"call {call}: max error {err.max():.3e} over the bound"
        assert np.array_equal(got, ref), f"call {call}: differs from qi_gemm_bf16 on the same device"
    torch.cuda.synchronize()


def test_noalloc_status_cleared_between_calls(qi):
    import torch
    from gpu_util import bf16_tensor
    M, N, K = 256, 256, 128
    A = bf16_tensor(synth.weight_bf16(34, 0, (M, K), std=1.0))
    B = bf16_tensor(synth.weight_bf16(34, 1, (N, K), std=1.0))
    first = _noalloc(qi, A, B, M, N, K, sync_check=0)
    torch.cuda.current_stream().synchronize()
    second = _noalloc(qi, A, B, M, N, K, sync_check=1)
    assert torch.equal(first, second)


def test_noalloc_rejects_oversize(qi):
    import torch
    A = torch.zeros(16, 64, dtype=torch.int16, device="cuda")
    st = qi.lib().qi_gemm_bf16_noalloc(A.data_ptr(), A.data_ptr(), A.data_ptr(), 32769, 256, 64, 1, None)
    assert st == 2
    assert b"above the limits 32768 x 24576 x 12288" in qi.lib().qi_last_error()
