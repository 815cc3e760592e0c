"""GPU parity of classifier-free guidance (qi_dit_step_cfg) against the oracle.

Two full-width blocks keep the oracle quick; the prompt lengths are 22 (the
256^2 workload's prompt) and 9 (the host contract's empty-prompt template).
"""
import numpy as np
import pytest

import synth
from oracle import dit as odit
from oracle import rope as orope
from oracle import sched as osched

from gpu_util import assert_close, f32_tensor, load_weights

pytestmark = pytest.mark.gpu

H = W = 16
N = H * W
L_POS, L_NEG = 22, 9
BLOCKS = 2


@pytest.fixture(scope="module")
def qi():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import diffusion_transformer_text_gb300 as q
    q.build()
    q.lib()
    return q


@pytest.fixture(scope="module")
def setup(qi):
    Wt = synth.Weights(seed=1, nblocks=BLOCKS)
    d = qi.DiT(blocks=BLOCKS, L_max=max(L_POS, L_NEG), N_max=N, kv_slots=2)
    load_weights(d, Wt)
    img = synth.input_f32(1, synth.J_IMG, (N, 64))
    prompts = {}
    for name, L, j in (("pos", L_POS, synth.J_TXT), ("neg", L_NEG, synth.J_TXT_LONG)):
        feats = synth.input_f32(1, j, (L, 4096))
        tabs = orope.token_tables(L, H, W)
        dev = dict(feats=f32_tensor(feats), L=L, txt_cos=f32_tensor(tabs[0]), txt_sin=f32_tensor(tabs[1]),
                   img_cos=f32_tensor(tabs[2]), img_sin=f32_tensor(tabs[3]))
        prompts[name] = (feats, tabs, dev)
    yield Wt, d, img, prompts
    d.close()


def test_cfg_step_matches_oracle(qi, setup):
    Wt, d, img, prompts = setup
    t, g = 0.83, 2.5
    vel = d.step_cfg(f32_tensor(img), t, g, prompts["pos"][2], prompts["neg"][2])
    d.check()
    ref = {}
    for name in ("pos", "neg"):
        feats, tabs, _ = prompts[name]
        ref[name] = odit.dit_forward(Wt, img, feats, np.float32(t), *tabs, nblocks=BLOCKS)
    assert_close(vel.cpu().numpy(), osched.cfg_combine(ref["pos"], ref["neg"], g), "guided velocity")


def test_cfg_cached_equals_joint(qi, setup):
    Wt, d, img, prompts = setup
    x = f32_tensor(synth.input_f32(1, 60, (N, 64)))
    joint = d.step_cfg(x, 0.5, 3.0, prompts["pos"][2], prompts["neg"][2]).clone()
    cached = d.step_cfg(x, 0.5, 3.0, prompts["pos"][2], prompts["neg"][2], use_cache=True)
    d.check()
    assert np.array_equal(joint.cpu().numpy(), cached.cpu().numpy())


def test_cfg_combine_is_the_stated_formula(qi, setup):
    """g = 0 gives the negative prompt's own velocity bit for bit; other g follow the
    oracle's float32 combine of the two single-prompt velocities exactly."""
    Wt, d, img, prompts = setup
    x = f32_tensor(img)
    pos = d.step(x, prompts["pos"][2]["feats"], 0.4, prompts["pos"][2]["txt_cos"], prompts["pos"][2]["txt_sin"],
                 prompts["pos"][2]["img_cos"], prompts["pos"][2]["img_sin"]).clone().cpu().numpy()
    neg = d.step(x, prompts["neg"][2]["feats"], 0.4, prompts["neg"][2]["txt_cos"], prompts["neg"][2]["txt_sin"],
                 prompts["neg"][2]["img_cos"], prompts["neg"][2]["img_sin"]).clone().cpu().numpy()
    v0 = d.step_cfg(x, 0.4, 0.0, prompts["pos"][2], prompts["neg"][2]).clone().cpu().numpy()
    v4 = d.step_cfg(x, 0.4, 4.0, prompts["pos"][2], prompts["neg"][2]).cpu().numpy()
    d.check()
    assert np.array_equal(v0, neg)
    assert v4.tobytes() == osched.cfg_combine(pos, neg, 4.0).tobytes()


def test_cfg_requires_two_slots(qi):
    d = qi.DiT(blocks=1, L_max=8, N_max=64)
    try:
        import torch
        z = torch.zeros(64, 64, device="cuda")
        tab = dict(feats=torch.zeros(8, 4096, device="cuda"), L=8, txt_cos=torch.zeros(8, 64, device="cuda"),
                   txt_sin=torch.zeros(8, 64, device="cuda"), img_cos=z, img_sin=z)
        with pytest.raises(qi.QiError) as e:
            d.step_cfg(z, 0.5, 2.0, tab, tab)
        assert e.value.status == 3
    finally:
        d.close()


def test_cfg_cached_is_one_batch2_pass_bit_exact(qi):
    """Cached guidance steps run both prompts' image rows in one pass of 2N rows. With
    N = 400 the second prompt starts inside a 128-row GEMM tile; each half must still
    equal that prompt's own image-only pass bit for bit, and the result the combine of
    the two."""
    import torch
    h = w = 20
    n = h * w
    Wt = synth.Weights(seed=1, nblocks=BLOCKS)
    d = qi.DiT(blocks=BLOCKS, L_max=max(L_POS, L_NEG), N_max=n, kv_slots=2)
    try:
        load_weights(d, Wt)
        prompts = {}
        for name, L, j in (("pos", L_POS, synth.J_TXT), ("neg", L_NEG, synth.J_TXT_LONG)):
            tabs = orope.token_tables(L, h, w)
            prompts[name] = dict(feats=f32_tensor(synth.input_f32(1, j, (L, 4096))), L=L,
                                 txt_cos=f32_tensor(tabs[0]), txt_sin=f32_tensor(tabs[1]),
                                 img_cos=f32_tensor(tabs[2]), img_sin=f32_tensor(tabs[3]))
        x = f32_tensor(synth.input_f32(1, 61, (n, 64)))
        d.step_cfg(x, 0.9, 3.0, prompts["pos"], prompts["neg"])                    # captures both
        guided = d.step_cfg(x, 0.6, 3.0, prompts["pos"], prompts["neg"], use_cache=True).cpu().numpy()
        single = {}
        for name in ("pos", "neg"):
            p = prompts[name]
            single[name] = d.step(x, p["feats"], 0.6, p["txt_cos"], p["txt_sin"], p["img_cos"],
                                  p["img_sin"]).cpu().numpy()
        d.check()
        assert guided.tobytes() == osched.cfg_combine(single["pos"], single["neg"], 3.0).tobytes()
        assert torch.isfinite(torch.from_numpy(guided)).all()
    finally:
        d.close()
