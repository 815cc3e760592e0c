"""GPU parity of the MXFP8 path: quantiser bit for bit, the block-scaled GEMM against
the exact product of the dequantised operands, and the block / pass in MXFP8 mode
against the oracle's MXFP8 block (oracle/mx.py)."""
import numpy as np
import pytest

import synth
from oracle import dit as odit
from oracle import mx as omx
from oracle import rope as orope

from gpu_util import assert_close, f32_tensor, load_weights, row_cos
# tolerances derived in test_oracle_mx.py from the library's fp16 operand roundings
from test_oracle_mx import MX_BLOCK_COS, MX_BLOCK_REL, MX_STEP_COS, MX_STEP_REL

RMS_RATIO = 0.75  # GPU-vs-MXFP8 rms error below this share of the MXFP8-vs-float32 difference


def _rms(a):
    return float(np.sqrt((np.asarray(a, np.float64) ** 2).mean()))

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


def _sf_bytes(sf, rows, K):
    """Scale bytes [rows, K/32] from the chunk layout (512-byte chunks [K/128][rows/128])."""
    G = (rows + 127) // 128
    r = np.arange(rows)[:, None]
    kb = np.arange(K // 32)[None, :]
    off = ((kb // 4) * G + r // 128) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + kb % 4
    return sf[off]


def _fp16_case(rows, K, seed):
    """fp16-exact values over many magnitudes, with an all-zero block, a saturating
    block and fp16 subnormals."""
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((rows, K)) * np.exp2(rng.integers(-14, 12, size=(rows, K // 32)).repeat(32, axis=1))
    r1, r2 = min(1, rows - 1), min(2, rows - 1)
    v[0, 0:32] = 0.0
    v[r1, 32:64] = 0.5
    v[r1, 40] = 500.0                                 # block max lands in [448, 512): clamps
    v[r2, 64:96] = rng.standard_normal(32) * 2.0 ** -20
    return v.astype(np.float16)


@pytest.mark.parametrize("rows,K", [(300, 512), (128, 128), (1, 4096)])
def test_quantiser_fp16_bit_exact(qi, rows, K):
    import torch
    h = _fp16_case(rows, K, rows + K)
    q, sf = qi.quant_mxfp8(torch.from_numpy(h).cuda(), bf16=False)
    ref_q, ref_e = omx.quantize(h.astype(np.float64))
    assert np.array_equal(q.cpu().numpy(), omx.e4m3_encode(ref_q))
    assert np.array_equal(_sf_bytes(sf.cpu().numpy(), rows, K), (ref_e + 127).astype(np.uint8))


def test_quantiser_bf16_weights_bit_exact(qi):
    import torch
    W = synth.Weights(seed=2, nblocks=1)
    w = W.block(0)["wo"][:384]                     # bf16 bits [384, 4096]
    q, sf = qi.quant_mxfp8(torch.from_numpy(w.view(np.int16)).cuda(), bf16=True)
    ref_q, ref_e = omx.quantize(odit.f32(w).astype(np.float64))
    assert np.array_equal(q.cpu().numpy(), omx.e4m3_encode(ref_q))
    assert np.array_equal(_sf_bytes(sf.cpu().numpy(), 384, 4096), (ref_e + 127).astype(np.uint8))


@pytest.mark.parametrize("M,N,K", [(300, 512, 512), (1000, 1024, 4096), (129, 256, 12288)])
def test_block_scaled_gemm(qi, M, N, K):
    """D = A B^T on MXFP8 operands equals the float64 product of the dequantised values
    to float32 accumulation error."""
    import torch
    d = qi.DiT(blocks=1, L_max=8, N_max=64)
    try:
        a = _fp16_case(M, K, 11)
        rng = np.random.default_rng(12)
        b = synth.f32_to_bf16_bits((rng.standard_normal((N, K)) * 0.02).astype(np.float32)).reshape(N, K)
        qa, sa = qi.quant_mxfp8(torch.from_numpy(a).cuda(), bf16=False)
        qb, sb = qi.quant_mxfp8(torch.from_numpy(b.view(np.int16)).cuda(), bf16=True)
        D = d.gemm_mxfp8(qa, sa, qb, sb, M, N, K)
        d.check()
        A = omx.dequantize(*omx.quantize(a.astype(np.float64)))
        B = omx.dequantize(*omx.quantize(odit.f32(b).astype(np.float64)))
        ref = A @ B.T
        got = D.cpu().numpy().astype(np.float64)
        scale = np.abs(A) @ np.abs(B).T                # error bound scale per element
        # one float32 rounding per K = 32 slice at most: (K / 32) * 2^-24 of the magnitude sum
        assert (np.abs(got - ref) <= (K / 32) * 2.0 ** -24 * scale + 1e-30).all(), np.abs(got - ref).max()
    finally:
        d.close()


def _mx_block_case():
    case = synth.BLOCK_CASE
    W = synth.Weights(seed=case.seed, nblocks=1)
    x = synth.block_hidden(case)
    tc, ts, ic, is_ = orope.token_tables(case.L, case.h, case.w)
    cos, sin = np.concatenate([tc, ic]), np.concatenate([ts, is_])
    mods = odit.row_mods(odit.modulation(W.glob, case.timestep), odit.modulation(W.glob, 0.0), case.L,
                         case.L + case.N)
    return case, W, x, cos, sin, mods


def test_one_block_mxfp8(qi):
    """The block in MXFP8 mode against the oracle's MXFP8 block. The GPU quantises fp16
    copies of the activations and runs attention on fp16 operands, so about 1 % of the
    E4M3 codes sit one step from the oracle's; the tolerance is derived from exactly
    those roundings, and the GPU must stay well inside the quantisation's own effect
    (the MXFP8 block against the float32 block)."""
    case, W, x, cos, sin, mods = _mx_block_case()
    d = qi.DiT(blocks=1, L_max=case.L, N_max=case.N, mxfp8=True)
    try:
        load_weights(d, W)
        d.set_mxfp8(True)
        got = d.block_forward(0, f32_tensor(x), case.L, case.timestep, f32_tensor(cos), f32_tensor(sin))
        d.check()
        got = got.cpu().numpy() - x
        ref = omx.block_forward(W.block(0), x, mods, case.L, cos, sin, 32) - x
        f32 = odit.block_forward(W.block(0), x, mods, case.L, cos, sin, 32) - x
        print(f"block: gpu-vs-mx rel {np.abs(got - ref).max() / np.abs(ref).max():.3e} cos "
              f"{row_cos(got, ref).min():.6f}; mx-vs-fp32 rel {np.abs(ref - f32).max() / np.abs(ref).max():.3e} "
              f"cos {row_cos(ref, f32).min():.6f}; rms ratio {_rms(got - ref) / _rms(ref - f32):.3f}", flush=True)
        assert_close(got, ref, "MXFP8 block update", cos_min=MX_BLOCK_COS, rel=MX_BLOCK_REL)
        assert _rms(got - ref) < RMS_RATIO * _rms(ref - f32)
        # the fp16 mode of the same handle is unchanged
        d.set_mxfp8(False)
        plain = d.block_forward(0, f32_tensor(x), case.L, case.timestep, f32_tensor(cos), f32_tensor(sin))
        assert_close(plain.cpu().numpy() - x, f32, "fp16 block update after switching back")
    finally:
        d.close()


def test_step_256_mxfp8_two_blocks(qi):
    case = synth.STEP_256
    nb = 2
    W = synth.Weights(seed=case.seed, nblocks=nb)
    d = qi.DiT(blocks=nb, L_max=case.L, N_max=case.N, mxfp8=True)
    try:
        load_weights(d, W)
        img = synth.img_tokens(case)
        txt = synth.txt_feats(case)
        tabs = orope.token_tables(case.L, case.h, case.w)
        dev = [f32_tensor(a) for a in tabs]
        d.set_mxfp8(True)
        vel = d.step(f32_tensor(img), f32_tensor(txt), case.timestep, *dev).clone()
        cached = d.step_cached(f32_tensor(img), case.L, case.timestep, dev[2], dev[3])
        d.check()
        got = vel.cpu().numpy()
        assert np.array_equal(got, cached.cpu().numpy())          # reuse stays exact in MXFP8 mode
        ref = omx.dit_forward(W, img, txt, np.float32(case.timestep), *tabs, nblocks=nb)
        f32 = odit.dit_forward(W, img, txt, np.float32(case.timestep), *tabs, nblocks=nb)
        print(f"step: gpu-vs-mx rel {np.abs(got - ref).max() / np.abs(ref).max():.3e} cos "
              f"{row_cos(got, ref).min():.6f}; mx-vs-fp32 rel {np.abs(ref - f32).max() / np.abs(ref).max():.3e} "
              f"cos {row_cos(ref, f32).min():.6f}; rms ratio {_rms(got - ref) / _rms(ref - f32):.3f}", flush=True)
        assert_close(got, ref, "MXFP8 velocity", cos_min=MX_STEP_COS, rel=MX_STEP_REL)
        assert _rms(got - ref) < RMS_RATIO * _rms(ref - f32)
    finally:
        d.close()


def test_mxfp8_requires_the_weight_copy(qi):
    d = qi.DiT(blocks=1, L_max=8, N_max=64)
    try:
        with pytest.raises(qi.QiError) as e:
            d.set_mxfp8(True)
        assert e.value.status == 3
    finally:
        d.close()


def test_mxfp8_guidance_batch2_bit_exact(qi):
    """MXFP8 mode with both prompts in one pass: the second prompt's attention output is
    quantised into the out-projection operand at a row offset (N = 400 starts it inside a
    128-row tile); each half must equal that prompt's own MXFP8 image-only pass."""
    from oracle import sched as osched
    h = w = 20
    n = h * w
    nb = 2
    Wt = synth.Weights(seed=1, nblocks=nb)
    d = qi.DiT(blocks=nb, L_max=22, N_max=n, kv_slots=2, mxfp8=True)
    try:
        load_weights(d, Wt)
        d.set_mxfp8(True)
        prompts = {}
        for name, L, j in (("pos", 22, synth.J_TXT), ("neg", 9, synth.J_TXT_LONG)):
            tabs = orope.token_tables(L, h, w)
            prompts[name] = dict(feats=f32_tensor(synth.input_f32(1, j, (L, 4096))), L=L,
                                 txt_cos=f32_tensor(tabs[0]), txt_sin=f32_tensor(tabs[1]),
                                 img_cos=f32_tensor(tabs[2]), img_sin=f32_tensor(tabs[3]))
        x = f32_tensor(synth.input_f32(1, 62, (n, 64)))
        d.step_cfg(x, 0.9, 2.0, prompts["pos"], prompts["neg"])
        guided = d.step_cfg(x, 0.5, 2.0, prompts["pos"], prompts["neg"], use_cache=True).cpu().numpy()
        single = {}
        for name in ("pos", "neg"):
            p = prompts[name]
            single[name] = d.step(x, p["feats"], 0.5, p["txt_cos"], p["txt_sin"], p["img_cos"],
                                  p["img_sin"]).cpu().numpy()
        d.check()
        assert guided.tobytes() == osched.cfg_combine(single["pos"], single["neg"], 2.0).tobytes()
    finally:
        d.close()
