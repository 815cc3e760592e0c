"""Failure detection on the GPU without faulting it: an allocation that fails is
reported as QI_ERR_OOM, a device wait that runs out (a barrier nothing arrives on,
bounded at 2 s) as QI_ERR_DEVICE_TIMEOUT, and in both cases the library keeps
working: the next call succeeds and reproduces the undisturbed result bit for bit."""
import time

import numpy as np
import pytest

import synth
from oracle import rope as orope

from gpu_util import f32_tensor, load_weights

pytestmark = pytest.mark.gpu

CASE = synth.BLOCK_CASE


@pytest.fixture(scope="module")
def qi():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import diffusion_transformer_text_gb300 as q
    q.build()
    q.lib()
    return q


def _inputs():
    img = synth.img_tokens(CASE)
    txt = synth.txt_feats(CASE)
    tabs = orope.token_tables(CASE.L, CASE.h, CASE.w)
    return img, txt, tabs


def test_allocation_failure_is_oom_and_recoverable(qi):
    for nth in (1, 2):                       # the weight store, then the activation store
        qi.debug_inject(1, nth)
        with pytest.raises(qi.QiError) as e:
            qi.DiT(blocks=1, L_max=CASE.L, N_max=CASE.N)
        assert e.value.status == 4
    d = qi.DiT(blocks=1, L_max=CASE.L, N_max=CASE.N)
    try:
        load_weights(d, synth.Weights(seed=CASE.seed, nblocks=1))
        img, txt, tabs = _inputs()
        vel = np.zeros((CASE.N, 64), np.float32)
        qi.debug_inject(1, 1)                # the first host-I/O staging buffer
        with pytest.raises(qi.QiError) as e:
            d.step_host(img, txt, CASE.L, 0.5, *tabs, vel)
        assert e.value.status == 4
        d.step_host(img, txt, CASE.L, 0.5, *tabs, vel)
        ref = d.step(f32_tensor(img), f32_tensor(txt), 0.5, *[f32_tensor(a) for a in tabs]).cpu().numpy()
        assert np.array_equal(vel, ref)
    finally:
        qi.debug_inject(0)
        d.close()


def test_device_wait_timeout_is_reported_and_recoverable(qi):
    d = qi.DiT(blocks=1, L_max=CASE.L, N_max=CASE.N)
    try:
        load_weights(d, synth.Weights(seed=CASE.seed, nblocks=1))
        img, txt, tabs = _inputs()
        args = (f32_tensor(img), f32_tensor(txt), 0.5, *[f32_tensor(a) for a in tabs])
        ref = d.step(*args).cpu().numpy()
        d.check()
        qi.debug_inject(2, dit=d)
        t0 = time.perf_counter()
        d.step(*args)
        with pytest.raises(qi.QiError) as e:
            d.check()
        waited = time.perf_counter() - t0
        assert e.value.status == 6
        assert 1.5 < waited < 60.0             # the wait ran into its 2 s bound, no longer
        d.check()                              # the report cleared the word
        again = d.step(*args).cpu().numpy()
        d.check()
        assert np.array_equal(again, ref)
    finally:
        qi.debug_inject(0, dit=d)
        d.close()
