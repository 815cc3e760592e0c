"""qi_gemm_bf16_noalloc: the GEMM for callers that may not allocate device memory.

Callers inside a host that owns all device memory (a fixed-arena inference
server, a plugin barred from the CUDA allocator) cannot create a qi_dit handle,
since creating one allocates. This entry point keeps its scratch (the kernel's
status word) in a static device array instead. The test calls it through the
C ABI twice in a row and checks each result against qi_gemm_bf16, the handle
path, with the same bound the GEMM tests use. It sits in its own file, collected
last, and needs nothing from earlier tests.
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


def _noalloc(qi, A, B, M, N, K):
    import torch
    D = torch.full((M, N), float("nan"), dtype=torch.float32, device=A.device)
    st = qi.lib().qi_gemm_bf16_noalloc(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, 1,
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, qi.lib().qi_last_error().decode()
    return D


def test_noalloc_matches_handle_gemm_twice(qi):
    from gpu_util import bf16_tensor
    d = qi.DiT(blocks=1, L_max=8, N_max=64)
    try:
        for M, N, K, seed in ((200, 512, 256, 31), (300, 768, 4096, 32)):
            A_bits = synth.weight_bf16(seed, 0, (M, K), std=1.0)
            B_bits = synth.weight_bf16(seed, 1, (N, K), std=1.0)
            A, B = bf16_tensor(A_bits), bf16_tensor(B_bits)
            ref = d.gemm(A, B).cpu().numpy()
            d.check()
            got = _noalloc(qi, A, B, M, N, K).cpu().numpy()
            a = synth.bf16_bits_to_f32(A_bits).astype(np.float64)
            b = synth.bf16_bits_to_f32(B_bits).astype(np.float64)
            bound = 1e-5 * (np.abs(a) @ np.abs(b).T) + 1e-6
            assert np.isfinite(got).all()
            assert (np.abs(got - ref) <= bound).all()
    finally:
        d.close()


def test_noalloc_rejects_oversize(qi):
    import torch
    A = torch.zeros(16, 64, dtype=torch.int16, device="cuda")
    st = qi.lib().qi_gemm_bf16_noalloc(A.data_ptr(), A.data_ptr(), A.data_ptr(), 16897, 256, 64, 1, None)
    assert st == 2
    assert b"above the limits" in qi.lib().qi_last_error()
