"""GPU parity of the individual kernels against the oracle, through the C ABI."""
import numpy as np
import pytest

import synth
from oracle import attention as oatt
from oracle import rope as orope
from oracle import sched as osched

from gpu_util import assert_close, bf16_tensor, f16_bits_to_f32, f16_tensor, f32_tensor

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


@pytest.fixture(scope="module")
def small_dit(qi):
    d = qi.DiT(blocks=1, L_max=16, N_max=64)
    yield d
    d.close()


# ---------------------------------------------------------------- GEMV

@pytest.mark.parametrize("in_dim,out_dim,silu_in", [(4096, 16384, True), (4096, 4096, True), (4096, 1000, False),
                                                    (4096, 100, True), (256, 4096, False)])
def test_gemv_matches_product(qi, in_dim, out_dim, silu_in):
    """The timestep / modulation GEMV (Core AI page, architecture table) against the
    float64 product of its bf16 weights and the oracle's activation, twice in a row
    (the streamed kernel's barriers start each call from phase 0); out_dim = 1000
    gives CTAs a partial last group of rows, out_dim = 100 fewer rows than SMs."""
    from oracle import dit as odit
    rng = np.random.default_rng(in_dim + out_dim)
    x = rng.standard_normal((2, in_dim)).astype(np.float32)
    W = synth.weight_bf16(41, out_dim, (out_dim, in_dim), std=0.02)
    b = synth.weight_bf16(42, out_dim, (out_dim,), std=0.02)
    act = odit.silu(x) if silu_in else x
    w64 = synth.bf16_bits_to_f32(W).astype(np.float64)
    exact = act.astype(np.float64) @ w64.T + synth.bf16_bits_to_f32(b).astype(np.float64)
    bound = 1e-5 * (np.abs(act).astype(np.float64) @ np.abs(w64).T) + 1e-6
    for call in range(2):
        y = qi.gemv(f32_tensor(x), bf16_tensor(W), bf16_tensor(b), silu_in).cpu().numpy()
        err = np.abs(y.astype(np.float64) - exact)
        assert (err <= bound).all(), f"call {call}: max error {err.max():.3e}"
    assert_close(y, odit.linear(act, W, b), f"gemv {in_dim}->{out_dim}")


# ---------------------------------------------------------------- GEMM

@pytest.mark.parametrize("M,N,K", [(1, 256, 64), (200, 512, 256), (300, 768, 4096), (129, 256, 12288)])
def test_gemm_matches_matmul(qi, small_dit, M, N, K):
    A = synth.weight_bf16(10, M, (M, K), std=1.0)
    B = synth.weight_bf16(11, N, (N, K), std=1.0)
    D = small_dit.gemm(bf16_tensor(A), bf16_tensor(B)).cpu().numpy()
    small_dit.check()
    a = synth.bf16_bits_to_f32(A).astype(np.float64)
    b = synth.bf16_bits_to_f32(B).astype(np.float64)
    ref = a @ b.T
    # bf16 products are exact in fp32; only the fp32 accumulation rounds. Bound the
    # error elementwise by a small multiple of sum_k |a_k b_k| (far below K * 2^-24).
    bound = 1e-5 * (np.abs(a) @ np.abs(b).T) + 1e-6
    assert (np.abs(D - ref) <= bound).all(), float((np.abs(D - ref) / bound).max())


@pytest.mark.parametrize("M,N,K", [
    (1024, 5120, 256),   # 80 pair tiles: a full wave, then the rest as 128-column halves
    (1024, 7424, 128),   # 116 tiles: the leftover fills more than half the pairs, stays whole
    (2048, 8192, 128),   # 256 tiles: several waves per pair, accumulator reuse, halves at the end
    (1000, 5120, 2048),  # ragged M (last pair half empty) over many k-blocks
])
def test_gemm_waves_and_tails(qi, small_dit, M, N, K):
    """Shapes with more 256 x 256 tiles than CTA pairs on a GB300 (152 SMs = 76 pairs), so the
    persistent schedule runs full tiles, repeated tiles per pair and the last-wave halves."""
    A = synth.weight_bf16(14, M, (M, K), std=1.0)
    B = synth.weight_bf16(15, N, (N, K), std=1.0)
    D = small_dit.gemm(bf16_tensor(A), bf16_tensor(B)).cpu().numpy()
    small_dit.check()
    a = synth.bf16_bits_to_f32(A).astype(np.float64)
    b = synth.bf16_bits_to_f32(B).astype(np.float64)
    ref = a @ b.T
    bound = 1e-5 * (np.abs(a) @ np.abs(b).T) + 1e-6
    assert (np.abs(D - ref) <= bound).all(), float((np.abs(D - ref) / bound).max())


def test_gemm_rows_independent_of_m(qi, small_dit):
    """A row's result does not depend on how many rows the pass has (exact)."""
    K = 4096
    A = synth.weight_bf16(12, 0, (300, K), std=1.0)
    B = synth.weight_bf16(13, 0, (512, K), std=1.0)
    full = small_dit.gemm(bf16_tensor(A), bf16_tensor(B)).cpu().numpy()
    part = small_dit.gemm(bf16_tensor(A[170:200]), bf16_tensor(B)).cpu().numpy()
    assert np.array_equal(full[170:200], part)


# ---------------------------------------------------------------- attention

def _qkv(R, seed):
    """fp16-valued q, k, v [R, 4096] (float32 arrays holding fp16 values)."""
    q = synth.normal_f32(seed, 0, R * 4096, np.float32(1.3)).astype(np.float16).astype(np.float32)
    k = synth.normal_f32(seed, 1, R * 4096, np.float32(1.3)).astype(np.float16).astype(np.float32)
    v = synth.normal_f32(seed, 2, R * 4096).astype(np.float16).astype(np.float32)
    return q.reshape(R, 4096), k.reshape(R, 4096), v.reshape(R, 4096)


def _oracle_att(q, k, v, L):
    R = q.shape[0]
    return oatt.attention_masked(q.reshape(R, 32, 128), k.reshape(R, 32, 128), v.reshape(R, 32, 128), L)


@pytest.mark.parametrize("L,N", [(7, 150), (1, 64), (130, 70), (22, 256)])
def test_attention_joint(qi, L, N):
    q, k, v = _qkv(L + N, L + N)
    o = qi.attention(f16_tensor(q), f16_tensor(k), f16_tensor(v), L)
    got = f16_bits_to_f32(o.cpu().numpy())
    ref = _oracle_att(q, k, v, L)
    assert_close(got.reshape(L + N, -1), ref, f"attention L={L} N={N}")


def test_attention_image_only_equals_joint(qi):
    """Image rows against stored text K/V give the joint pass's image rows bit for bit."""
    L, N = 37, 200
    q, k, v = _qkv(L + N, 5)
    qt, kt, vt = f16_tensor(q), f16_tensor(k), f16_tensor(v)
    joint = qi.attention(qt, kt, vt, L).cpu().numpy()
    img = qi.attention(qt[L:].contiguous(), kt, vt, L, q_off=L).cpu().numpy()
    assert np.array_equal(joint[L:], img)
    # and the text rows of a text-only pass equal the joint pass's text rows
    txt = qi.attention(qt[:L].contiguous(), kt[:L].contiguous(), vt[:L].contiguous(), L).cpu().numpy()
    assert np.array_equal(joint[:L], txt)


def test_attention_consecutive_short_units(qi):
    """A CTA that runs several one-key-tile units in a row: with 2400 query rows a head
    has 19 row units, so on 152 SMs (608 units, 4 per CTA) a CTA whose first unit is a
    head's rows 0..127 gets the first units of four heads; with L = 400 those rows are
    text rows whose keys end inside the first key tile. Each unit's row sums must not be
    overwritten before the previous unit's output is stored. Sampled rows against the
    oracle: the first unit's, other text rows, and image rows."""
    L, N = 400, 2000
    R = L + N
    q, k, v = _qkv(R, 17)
    o = qi.attention(f16_tensor(q), f16_tensor(k), f16_tensor(v), L)
    got = f16_bits_to_f32(o.cpu().numpy())
    rows = np.array([0, 1, 31, 64, 127, 128, 200, 255, 399, 400, 401, 1200, 2047, R - 1])
    ref = oatt.attention_rows(q[rows].reshape(len(rows), 32, 128), rows, k.reshape(R, 32, 128),
                              v.reshape(R, 32, 128), L)
    assert_close(got[rows], ref, "attention L=400 N=2000 sampled rows")


def test_attention_long_keys(qi):
    """Several query and key tiles with a ragged tail at a realistic head count."""
    L, N = 407, 600
    q, k, v = _qkv(L + N, 9)
    o = qi.attention(f16_tensor(q), f16_tensor(k), f16_tensor(v), L)
    got = f16_bits_to_f32(o.cpu().numpy())
    assert_close(got, _oracle_att(q, k, v, L), "attention 407+600")


# ---------------------------------------------------------------- RoPE, Euler, packing

def test_rope_axis_tables_bit_exact(qi):
    got = qi.rope_axis_tables(10000.0)
    ref = orope.axis_tables()
    for (gc, gs), (rc, rs) in zip(got, ref):
        assert np.array_equal(gc.cpu().numpy(), rc)
        assert np.array_equal(gs.cpu().numpy(), rs)


@pytest.mark.parametrize("L,h,w", [(8, 8, 8), (22, 16, 16), (407, 64, 64), (512, 128, 128), (3, 5, 7)])
def test_rope_token_tables_bit_exact(qi, L, h, w):
    got = [t.cpu().numpy() for t in qi.rope_tables(L, h, w)]
    ref = orope.token_tables(L, h, w)
    for g, r in zip(got, ref):
        assert g.tobytes() == r.tobytes()


@pytest.mark.parametrize("N", [1, 255, 4096])
def test_euler_bit_exact(qi, N):
    x = synth.input_f32(3, 50, (N, 64))
    v = synth.input_f32(3, 51, (N, 64))
    s, _ = osched.flow_sigmas(40, 4096)
    xt = f32_tensor(x)
    qi.euler_update(xt, f32_tensor(v), float(s[7]), float(s[8]))
    assert xt.cpu().numpy().tobytes() == osched.euler_update(x, v, s[7], s[8]).tobytes()


@pytest.mark.parametrize("N", [64, 4096, 16384])
def test_dpmpp2m_loop_bit_exact(qi, N):
    """A whole 40-step DPM++ 2M loop (orders 1, 1, 2 ... 2, 0) over a velocity that
    changes every step, against the oracle; every step's x and carried D bit for bit."""
    import torch
    s, _ = osched.flow_sigmas(40, N)
    x = synth.input_f32(6, 52, (N, 64))
    xt = f32_tensor(x)
    dt = torch.full((N, 64), float("nan"), device="cuda")   # contents before step 0 are never read
    dp = None
    for i in range(40):
        v = (synth.input_f32(6, 100 + i, (N, 64)) + 0.5 * x).astype(np.float32)
        x, dp = osched.dpmpp2m_update(x, v, dp, s, i)
        qi.dpmpp2m_update(xt, f32_tensor(v), dt, s, i)
        if i in (0, 1, 2, 20, 39):
            assert xt.cpu().numpy().tobytes() == x.tobytes(), i
            assert dt.cpu().numpy().tobytes() == dp.tobytes(), i
    assert xt.cpu().numpy().tobytes() == x.tobytes()


@pytest.mark.parametrize("h,w", [(8, 8), (64, 64), (5, 3)])
def test_pack_noise_exact(qi, h, w):
    z = synth.input_f32(4, 2, (64, h, w))
    x = qi.pack_noise(f32_tensor(z)).cpu().numpy()
    assert np.array_equal(x, orope.pack_noise(z))
