"""GPU parity of the DiT block and the full step against the oracle (C ABI)."""
import numpy as np
import pytest

import synth
from oracle import dit as odit
from oracle import rope as orope

from gpu_util import assert_close, check_ranges, f16_bits_to_f32, f32_tensor, load_weights, range_buffer

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


def _tables(L, h, w):
    tc, ts, ic, is_ = orope.token_tables(L, h, w)
    return tc, ts, ic, is_


# ---------------------------------------------------------------- one block

def test_one_block(qi):
    """One block at full width: hidden [72, 4096], L = 8 text rows then an 8x8 grid."""
    case = synth.BLOCK_CASE
    W = synth.Weights(seed=case.seed, nblocks=1)
    d = qi.DiT(blocks=1, L_max=case.L, N_max=case.N)
    try:
        load_weights(d, W)
        x = synth.block_hidden(case)
        tc, ts, ic, is_ = _tables(case.L, case.h, case.w)
        cos, sin = np.concatenate([tc, ic]), np.concatenate([ts, is_])
        mods = odit.row_mods(odit.modulation(W.glob, case.timestep), odit.modulation(W.glob, 0.0), case.L,
                             case.L + case.N)
        ref, rk, rv = odit.block_forward(W.block(0), x, mods, case.L, cos, sin, 32, return_kv=True)
        got = d.block_forward(0, f32_tensor(x), case.L, case.timestep, f32_tensor(cos), f32_tensor(sin))
        d.check()
        got = got.cpu().numpy()
        # the residual carries the input through; judge the block's update
        assert_close(got - x, ref - x, "block update")
        k, v = d.read_kv(0, 0, case.L + case.N)
        k = f16_bits_to_f32(k.cpu().numpy())
        v = f16_bits_to_f32(v.cpu().numpy())
        assert_close(k, rk.reshape(case.L + case.N, -1), "stored K (post-RoPE)")
        assert_close(v, rv.reshape(case.L + case.N, -1), "stored V")
    finally:
        d.close()


# ---------------------------------------------------------------- full step, 256^2

@pytest.fixture(scope="module")
def dit256(qi):
    case = synth.STEP_256
    W = synth.Weights(seed=case.seed)
    d = qi.DiT(blocks=32, L_max=case.L, N_max=case.N)
    load_weights(d, W)
    yield case, W, d
    d.close()


def test_profile_classes_selects_kernel_classes(qi, dit256):
    """Class-selective timing: only the named classes record launches (one gate/up GEMM
    per block, or per fourth block with a stride of 4), every class when enabled without
    names, nothing when off; a mask bit past the last class or a stride below 1 is
    rejected."""
    case, W, d = dit256
    img = f32_tensor(synth.img_tokens(case))
    txt = f32_tensor(synth.txt_feats(case))
    tabs = [f32_tensor(a) for a in _tables(case.L, case.h, case.w)]
    d.profile(True, classes=["gateup_gemm"])
    d.step(img, txt, case.timestep, *tabs)
    prof = d.profile_read()
    assert prof["gateup_gemm"][1] == 32 and prof["gateup_gemm"][0] > 0
    assert all(n == 0 for c, (_, n) in prof.items() if c != "gateup_gemm")
    d.profile(True, classes=["gateup_gemm", "attention"], block_stride=4)
    d.step(img, txt, case.timestep, *tabs)
    prof = d.profile_read()
    assert prof["gateup_gemm"][1] == 8 and prof["attention"][1] == 8
    assert all(n == 0 for c, (_, n) in prof.items() if c not in ("gateup_gemm", "attention"))
    d.profile(True)
    d.step(img, txt, case.timestep, *tabs)
    prof = d.profile_read()
    assert all(n > 0 for _, n in prof.values())
    d.profile(False)
    d.step(img, txt, case.timestep, *tabs)
    assert all(n == 0 for _, n in d.profile_read().values())
    assert qi.lib().qi_dit_profile_classes(d._h, 1 << len(qi.PROF_CLASSES), 1) == 1
    assert qi.lib().qi_dit_profile_classes(d._h, 8, 0) == 1
    d.check()


def test_step_256(qi, dit256):
    case, W, d = dit256
    img = synth.img_tokens(case)
    txt = synth.txt_feats(case)
    tc, ts, ic, is_ = _tables(case.L, case.h, case.w)
    rb = range_buffer(d)
    d.set_range_probe(rb)
    vel = d.step(f32_tensor(img), f32_tensor(txt), case.timestep, f32_tensor(tc), f32_tensor(ts), f32_tensor(ic),
                 f32_tensor(is_))
    d.set_range_probe(None)
    d.check()
    ref = odit.dit_forward(W, img, txt, np.float32(case.timestep), tc, ts, ic, is_)
    assert_close(vel.cpu().numpy(), ref, "vel 256^2")
    check_ranges(rb.cpu().numpy(), "256^2 joint step")


def test_reuse_equals_joint_bit_exact(qi, dit256):
    """Image-only steps over the captured text K/V reproduce the joint pass exactly."""
    case, W, d = dit256
    img = f32_tensor(synth.img_tokens(case))
    txt = f32_tensor(synth.txt_feats(case))
    tc, ts, ic, is_ = [f32_tensor(a) for a in _tables(case.L, case.h, case.w)]
    for t in (0.97, 0.41):
        joint = d.step(img, txt, t, tc, ts, ic, is_).clone()
        cached = d.step_cached(img, case.L, t, ic, is_)
        d.check()
        assert np.array_equal(joint.cpu().numpy(), cached.cpu().numpy())
    # a different image at another t still matches its own joint pass
    img2 = f32_tensor(synth.input_f32(case.seed, 77, (case.N, 64)))
    c2 = d.step_cached(img2, case.L, 0.2, ic, is_).clone()
    j2 = d.step(img2, txt, 0.2, tc, ts, ic, is_)
    assert np.array_equal(c2.cpu().numpy(), j2.cpu().numpy())


def test_euler_step_equals_step_then_update(qi, dit256):
    """qi_dit_euler_step (device and host buffers) = qi_dit_step then qi_euler_update, bit for bit,
    for a joint step and a cached step; the host call returns x and vel in the caller's buffers."""
    import torch
    case, W, d = dit256
    sig, ts_ = qi.flow_sigmas(40, case.N)
    img0 = synth.img_tokens(case)
    txt = synth.txt_feats(case)
    tabs = _tables(case.L, case.h, case.w)
    tc, ts, ic, is_ = [f32_tensor(a) for a in tabs]
    txt_d = f32_tensor(txt)
    for i, use_cache in ((0, False), (1, True)):
        t = float(np.float32(ts_[i]) / np.float32(1000.0))
        # reference: the two calls
        x_ref = f32_tensor(img0)
        if use_cache:
            v_ref = d.step_cached(x_ref, case.L, t, ic, is_).clone()
        else:
            v_ref = d.step(x_ref, txt_d, t, tc, ts, ic, is_).clone()
        qi.euler_update(x_ref, v_ref, float(sig[i]), float(sig[i + 1]))
        # device sampler step
        x_dev = f32_tensor(img0)
        v_dev = torch.empty_like(x_dev)
        d.euler_step(x_dev, None if use_cache else txt_d, case.L, t, float(sig[i]), float(sig[i + 1]),
                     None if use_cache else tc, None if use_cache else ts, ic, is_, use_cache=use_cache, vel=v_dev)
        # host sampler step (pinned buffers), and with vel_out NULL
        x_h = torch.from_numpy(img0.copy()).pin_memory()
        v_h = torch.empty(case.N, 64).pin_memory()
        host = [torch.from_numpy(np.ascontiguousarray(a)).pin_memory() for a in tabs]
        txt_h = torch.from_numpy(txt.copy()).pin_memory()
        d.euler_step_host(x_h, txt_h, case.L, t, float(sig[i]), float(sig[i + 1]), host[0], host[1], host[2], host[3],
                          use_cache=use_cache, vel=v_h)
        x_n = img0.copy()
        d.euler_step_host(x_n, None if use_cache else txt, case.L, t, float(sig[i]), float(sig[i + 1]),
                          None if use_cache else np.ascontiguousarray(tabs[0]),
                          None if use_cache else np.ascontiguousarray(tabs[1]), np.ascontiguousarray(tabs[2]),
                          np.ascontiguousarray(tabs[3]), use_cache=use_cache)
        d.check()
        xr, vr = x_ref.cpu().numpy(), v_ref.cpu().numpy()
        assert np.array_equal(x_dev.cpu().numpy(), xr) and np.array_equal(v_dev.cpu().numpy(), vr)
        assert np.array_equal(x_h.numpy(), xr) and np.array_equal(v_h.numpy(), vr)
        assert np.array_equal(x_n, xr)
        assert not np.array_equal(xr, img0)


def test_text_only_capture_equals_joint(qi, dit256):
    """A text-only pass stores the same text K/V as a joint pass, bit for bit."""
    case, W, d = dit256
    img = f32_tensor(synth.img_tokens(case))
    txt = f32_tensor(synth.txt_feats(case))
    tc, ts, ic, is_ = [f32_tensor(a) for a in _tables(case.L, case.h, case.w)]
    d.step(img, txt, 0.97, tc, ts, ic, is_)
    joint = [tuple(t.cpu().numpy() for t in d.read_kv(b, 0, case.L)) for b in (0, 13, 31)]
    d.text_kv_capture(txt, tc, ts)
    d.check()
    for (jk, jv), b in zip(joint, (0, 13, 31)):
        k, v = d.read_kv(b, 0, case.L)
        assert np.array_equal(jk, k.cpu().numpy()) and np.array_equal(jv, v.cpu().numpy())


def test_weight_outside_fp16_range_is_rejected(qi):
    """Tensor-core weights are kept as fp16: a bf16 value beyond +-65504 fails the load."""
    d = qi.DiT(blocks=1, L_max=8, N_max=64)
    try:
        W = synth.Weights(seed=0, nblocks=1)
        g = dict(W.glob)
        txt_w = g["txt_w"].copy()
        txt_w[5, 7] = synth.f32_to_bf16_bits(np.array([1.0e5], np.float32))[0]
        g["txt_w"] = txt_w
        with pytest.raises(qi.QiError) as e:
            d.load_global(g)
        assert e.value.status == 1 and "fp16 range" in str(e.value)
        bw = dict(W.block(0))
        wd = bw["wd"].copy()
        wd[0, 0] = synth.f32_to_bf16_bits(np.array([-7.0e4], np.float32))[0]
        bw["wd"] = wd
        with pytest.raises(qi.QiError) as e:
            d.load_block(0, bw)
        assert e.value.status == 1
    finally:
        d.close()


def test_nonfinite_velocity_is_reported(qi):
    """A NaN planted in a bias reaches the velocity; the head's guard reports it."""
    case = synth.BLOCK_CASE
    d = qi.DiT(blocks=1, L_max=case.L, N_max=case.N)
    try:
        W = synth.Weights(seed=0, nblocks=1)
        g = dict(W.glob)
        img_b = g["img_b"].copy()
        img_b[3] = 0x7FC0  # bf16 quiet NaN
        g["img_b"] = img_b
        d.load_global(g)
        d.load_block(0, W.block(0))
        tc, ts, ic, is_ = [f32_tensor(a) for a in _tables(case.L, case.h, case.w)]
        d.step(f32_tensor(synth.img_tokens(case)), f32_tensor(synth.txt_feats(case)), 0.5, tc, ts, ic, is_)
        with pytest.raises(qi.QiError) as e:
            d.check()
        assert e.value.status == 8
        d.check()  # the word was cleared by the report
    finally:
        d.close()


def test_fp16_overflow_of_h_is_reported(qi):
    """SwiGLU weights scaled by 128 (exact in bf16) push h far past fp16's 65504. The fp32
    oracle shows the overflow is real and its velocity stays finite; the library, whose
    down-GEMM input is fp16, must report QI_ERR_NONFINITE rather than return a finite
    wrong velocity, and the range probe must see the overflow."""
    case = synth.BLOCK_CASE
    W = synth.Weights(seed=0, nblocks=1)
    bw = dict(W.block(0))
    for k in ("wg", "wu"):
        bw[k] = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(bw[k]) * np.float32(128.0)).reshape(bw[k].shape)
    W._blocks[0] = bw
    img, txt = synth.img_tokens(case), synth.txt_feats(case)
    tc, ts, ic, is_ = _tables(case.L, case.h, case.w)
    t = np.float32(case.timestep)
    # oracle: h of block 0 in fp32
    R = case.L + case.N
    mods = odit.row_mods(odit.modulation(W.glob, t), odit.modulation(W.glob, 0.0), case.L, R)
    s1, g1, s2, g2 = odit.mod_chunks(mods)
    cos, sin = np.concatenate([tc, ic]), np.concatenate([ts, is_])
    x = odit.embed(W.glob, img, txt)
    q, k, v = odit.block_qkv(bw, x, s1, cos, sin, 32)
    from oracle.attention import attention_masked
    o = attention_masked(q, k, v, case.L)
    x1 = x + g1 * odit.linear(o.reshape(R, -1), bw["wo"])
    xn2 = odit.rmsnorm(x1) * (np.float32(1.0) + s2)
    h = odit.silu(odit.linear(xn2, bw["wg"])) * odit.linear(xn2, bw["wu"])
    assert np.abs(h).max() > 4 * 65504.0
    ref = odit.dit_forward(W, img, txt, t, tc, ts, ic, is_, nblocks=1)
    assert np.isfinite(ref).all()
    # library
    d = qi.DiT(blocks=1, L_max=case.L, N_max=case.N)
    try:
        d.load_global(W.glob)
        d.load_block(0, bw)
        rb = range_buffer(d)
        d.set_range_probe(rb)
        d.step(f32_tensor(img), f32_tensor(txt), float(t), f32_tensor(tc), f32_tensor(ts), f32_tensor(ic),
               f32_tensor(is_))
        d.set_range_probe(None)
        with pytest.raises(qi.QiError) as e:
            d.check()
        assert e.value.status == 8
        r = rb.cpu().numpy()
        assert np.isinf(r[0, qi.RANGE_KINDS.index("h")])
        assert np.isfinite(r[0, :qi.RANGE_KINDS.index("h")]).all()
    finally:
        d.close()


def test_use_cache_requires_capture(qi):
    d = qi.DiT(blocks=1, L_max=8, N_max=64)
    try:
        import torch
        img = torch.zeros(64, 64, device="cuda")
        cs = torch.zeros(64, 64, device="cuda")
        W = synth.Weights(seed=0, nblocks=1)
        load_weights(d, W)
        with pytest.raises(qi.QiError) as e:
            d.step_cached(img, 8, 0.5, cs, cs)
        assert e.value.status == 3
    finally:
        d.close()


# ---------------------------------------------------------------- degenerate and ragged shapes

@pytest.mark.parametrize("L,h,w", [(1, 1, 1), (1, 1, 2), (3, 5, 3), (130, 3, 7)])
def test_step_small_and_ragged_shapes(qi, L, h, w):
    """One-token prompts, one-token images, non-square grids and a prompt longer than the
    image: the two-block pass against the oracle, reuse bit-exact, capture exact."""
    N = h * w
    nb = 2
    W = synth.Weights(seed=9, nblocks=nb)
    d = qi.DiT(blocks=nb, L_max=L, N_max=N)
    try:
        load_weights(d, W)
        img = synth.input_f32(9, 0, (N, 64))
        txt = synth.input_f32(9, 1, (L, 4096))
        tc, ts, ic, is_ = _tables(L, h, w)
        dev = [f32_tensor(a) for a in (tc, ts, ic, is_)]
        vel = d.step(f32_tensor(img), f32_tensor(txt), 0.7, *dev).clone()
        cached = d.step_cached(f32_tensor(img), L, 0.7, dev[2], dev[3])
        d.check()
        ref = odit.dit_forward(W, img, txt, np.float32(0.7), tc, ts, ic, is_, nblocks=nb)
        assert_close(vel.cpu().numpy(), ref, f"L={L} {h}x{w}")
        assert np.array_equal(vel.cpu().numpy(), cached.cpu().numpy())
        joint_kv = [t.cpu().numpy() for t in d.read_kv(1, 0, L)]
        d.text_kv_capture(f32_tensor(txt), dev[0], dev[1])
        d.check()
        cap_kv = [t.cpu().numpy() for t in d.read_kv(1, 0, L)]
        assert all(np.array_equal(a, b) for a, b in zip(joint_kv, cap_kv))
    finally:
        d.close()


def test_step_rejects_out_of_range_shapes(qi):
    d = qi.DiT(blocks=1, L_max=8, N_max=64)
    try:
        import torch
        W = synth.Weights(seed=0, nblocks=1)
        load_weights(d, W)
        L = qi.lib()
        z = lambda r, c: torch.zeros(r, c, device="cuda")
        vel = z(128, 64)
        for N, Lq in ((0, 8), (65, 8), (64, 0), (64, 9)):
            st = L.qi_dit_step(d._h, z(max(N, 1), 64).data_ptr(), N, z(max(Lq, 1), 4096).data_ptr(), Lq, 0.5,
                               z(max(Lq, 1), 64).data_ptr(), z(max(Lq, 1), 64).data_ptr(),
                               z(max(N, 1), 64).data_ptr(), z(max(N, 1), 64).data_ptr(), vel.data_ptr(), 0, None)
            assert st == 2, (N, Lq, st)
        st = L.qi_dit_step(d._h, z(64, 64).data_ptr(), 64, z(8, 4096).data_ptr(), 8, float("nan"),
                           z(8, 64).data_ptr(), z(8, 64).data_ptr(), z(64, 64).data_ptr(), z(64, 64).data_ptr(),
                           vel.data_ptr(), 0, None)
        assert st == 1
        d.check()
    finally:
        d.close()
