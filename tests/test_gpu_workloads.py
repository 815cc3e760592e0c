"""GPU parity on the three full-size workloads, in the launch configuration the bench uses.

* 384^2 (N = 576), a 22-token then a 494-token prompt: step 1 is the joint pass that
  captures the text K/V, steps 2-5 run image rows over the stored K/V. Every cached
  step equals a full joint recomputation bit for bit; step 1 (both prompts) and
  step 5 (494 tokens, teacher-forced) match the dense oracle pass.
* 1024^2 (N = 4096, L = 407), the whole 40-step FlowMatch Euler loop: sigmas and
  every checked Euler update bit-exact, cached steps equal joint recomputation, and
  at steps 0, 20 and 39 sampled rows of blocks 0, 15, 31, of the embedding and of
  the head match the oracle, teacher-forced from the residual stream the GPU traced.
* 2048^2 (N = 16384, L = 512): one joint step and one cached step, the same checks.

The oracle evaluates a block for selected rows (all rows' K/V, then the chosen
queries); that is the dense definition restricted to those rows.
"""
import numpy as np
import pytest

import synth
from oracle import dit as odit
from oracle import rope as orope
from oracle import sched as osched

from gpu_util import assert_close, check_ranges, f32_tensor, load_weights, range_buffer

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
    return [f32_tensor(a) for a in orope.token_tables(L, h, w)], orope.token_tables(L, h, w)


def _t(ts, i):
    return float(osched.dit_timestep(ts, i))


def _sample_rows(L, N, seed, n_img=24):
    rng = np.random.default_rng(seed)
    txt = sorted({0, 1, L // 2, L - 1})
    img = sorted({0, N - 1, N // 2} | set(rng.choice(N, n_img, replace=False).tolist()))
    return np.array(txt), np.array(img)


class Tracer:
    """Runs a step with the residual stream traced around one block."""

    def __init__(self, qi, d, R):
        import torch
        self.d = d
        self.a = torch.empty(R, 4096, device="cuda")
        self.b = torch.empty(R, 4096, device="cuda")

    def around(self, block, run):
        self.d.set_trace(0, block, self.a)
        self.d.set_trace(1, block + 1, self.b)
        run()
        self.d.set_trace(0, 0, None)
        self.d.set_trace(1, 0, None)
        self.d.check()
        return self.a.cpu().numpy(), self.b.cpu().numpy()

    def at(self, block, run):
        self.d.set_trace(0, block, self.a)
        run()
        self.d.set_trace(0, 0, None)
        self.d.check()
        return self.a.cpu().numpy()


# ---------------------------------------------------------------- 384^2, two prompts


def test_384_two_prompts_reuse(qi):
    h = w = 24
    N = h * w
    W = synth.Weights(seed=synth.STEP_384_L22.seed)
    d = qi.DiT(blocks=32, L_max=494, N_max=N)
    try:
        load_weights(d, W)
        sig, ts = qi.flow_sigmas(40, N)
        z = synth.noise_latent(synth.STEP_384_L22)
        for L, j in ((22, synth.J_TXT), (494, synth.J_TXT_LONG)):
            txt_np = synth.input_f32(2, j, (L, 4096))
            txt = f32_tensor(txt_np)
            (tc, tsn, ic, isn), (otc, ots, oic, ois) = _tables(L, h, w)
            x = qi.pack_noise(f32_tensor(z))
            assert np.array_equal(x.cpu().numpy(), orope.pack_noise(z))
            for i in range(5):
                t = _t(ts, i)
                if i == 0:
                    rb = range_buffer(d)
                    d.set_range_probe(rb)
                    vel = d.step(x, txt, t, tc, tsn, ic, isn).clone()
                    d.set_range_probe(None)
                    check_ranges(rb.cpu().numpy(), f"384^2 L={L} joint step 1")
                    ref = odit.dit_forward(W, x.cpu().numpy(), txt_np, np.float32(t), otc, ots, oic, ois)
                    assert_close(vel.cpu().numpy(), ref, f"384^2 L={L} step 1 vs oracle")
                else:
                    if i == 4:
                        rb = range_buffer(d)
                        d.set_range_probe(rb)
                    vel = d.step_cached(x, L, t, ic, isn).clone()
                    if i == 4:
                        d.set_range_probe(None)
                        check_ranges(rb.cpu().numpy(), f"384^2 L={L} cached step 5")
                    joint = d.step(x, txt, t, tc, tsn, ic, isn)
                    assert np.array_equal(vel.cpu().numpy(), joint.cpu().numpy()), f"L={L} step {i + 1}"
                    if i == 4 and L == 494:
                        ref = odit.dit_forward(W, x.cpu().numpy(), txt_np, np.float32(t), otc, ots, oic, ois)
                        assert_close(vel.cpu().numpy(), ref, f"384^2 L={L} step 5 (teacher-forced) vs oracle")
                x_before = x.cpu().numpy()
                qi.euler_update(x, vel, float(sig[i]), float(sig[i + 1]))
                assert x.cpu().numpy().tobytes() == osched.euler_update(
                    x_before, vel.cpu().numpy(), sig[i], sig[i + 1]).tobytes()
            d.check()
    finally:
        d.close()


# ---------------------------------------------------------------- shared sampled checks


def _check_embed(W, trace0, img_np, txt_np, rows_txt, rows_img, L, what):
    ref = odit.embed(W.glob, img_np[rows_img], txt_np[rows_txt] if len(rows_txt) else txt_np[:0])
    got = np.concatenate([trace0[rows_txt], trace0[L + rows_img]]) if len(rows_txt) else trace0[rows_img]
    assert_close(got, ref, what)


def _check_block(W, b, x_all, x_out_rows, mods, L, cos, sin, rows, what):
    ref, _ = odit.block_forward_rows(W.block(b), x_all, mods, L, cos, sin, 32, rows)
    assert_close(x_out_rows - x_all[rows], ref - x_all[rows], what)


def _check_head(W, x_final_img, vel, rows_img, what):
    ref = odit.head(W.glob, x_final_img[rows_img])
    assert_close(vel[rows_img], ref, what)


# ---------------------------------------------------------------- 1024^2, 40 steps


def test_1024_forty_step_loop(qi):
    case = synth.LOOP_1024
    L, h, w = case.L, case.h, case.w
    N = h * w
    R = L + N
    W = synth.Weights(seed=case.seed)
    d = qi.DiT(blocks=32, L_max=L, N_max=N)
    try:
        load_weights(d, W)
        sig, ts = qi.flow_sigmas(40, N)
        rs, rt = osched.flow_sigmas(40, N)
        assert sig.tobytes() == rs.tobytes() and ts.tobytes() == rt.tobytes()
        txt_np = synth.txt_feats(case)
        txt = f32_tensor(txt_np)
        (tc, tsn, ic, isn), (otc, ots, oic, ois) = _tables(L, h, w)
        cos, sin = np.concatenate([otc, oic]), np.concatenate([ots, ois])
        z = synth.noise_latent(case)
        x = qi.pack_noise(f32_tensor(z))
        tr = Tracer(qi, d, R)
        rows_txt, rows_img = _sample_rows(L, N, seed=40)
        text_x = {}
        checked = 0
        for i in range(40):
            t = _t(ts, i)
            if i == 0:
                run = lambda: d.step(x, txt, t, tc, tsn, ic, isn)
            else:
                run = lambda: d.step_cached(x, L, t, ic, isn)
            if i in (0, 20, 39):
                mods = odit.row_mods(odit.modulation(W.glob, np.float32(t)), odit.modulation(W.glob, 0.0), L, R)
                x_np = x.cpu().numpy()
                for b in (0, 15, 31):
                    a_, b_ = tr.around(b, run)
                    if i == 0:
                        text_x[b] = a_[:L].copy()
                        x_all, out = a_[:R], b_[:R]
                        rows = np.concatenate([rows_txt, L + rows_img])
                        got = out[rows]
                    else:
                        x_all = np.concatenate([text_x[b], a_[:N]])
                        rows = L + rows_img
                        got = b_[:N][rows_img]
                    _check_block(W, b, x_all, got, mods, L, cos, sin, rows, f"1024^2 step {i} block {b}")
                    checked += 1
                if i == 0:
                    _check_embed(W, tr.at(0, run), x_np, txt_np, rows_txt, rows_img, L, "1024^2 embedding")
                x_fin = tr.at(32, run)
                rb = range_buffer(d)
                d.set_range_probe(rb)
                vel = run().clone()
                d.set_range_probe(None)
                check_ranges(rb.cpu().numpy(), f"1024^2 step {i} ({'joint' if i == 0 else 'cached'})")
                _check_head(W, x_fin[L:R] if i == 0 else x_fin[:N], vel.cpu().numpy(), rows_img,
                            f"1024^2 step {i} head")
                if i > 0:
                    joint = d.step(x, txt, t, tc, tsn, ic, isn)
                    assert np.array_equal(vel.cpu().numpy(), joint.cpu().numpy()), f"step {i} reuse"
                x_before = x_np
                qi.euler_update(x, vel, float(sig[i]), float(sig[i + 1]))
                assert x.cpu().numpy().tobytes() == osched.euler_update(
                    x_before, vel.cpu().numpy(), sig[i], sig[i + 1]).tobytes()
            else:
                vel = run()
                qi.euler_update(x, vel, float(sig[i]), float(sig[i + 1]))
        d.check()
        assert checked == 9
        assert np.isfinite(x.cpu().numpy()).all()
    finally:
        d.close()


# ---------------------------------------------------------------- 2048^2


def test_2048_step(qi):
    case = synth.STEP_2048
    L, h, w = case.L, case.h, case.w
    N = h * w
    R = L + N
    W = synth.Weights(seed=case.seed)
    d = qi.DiT(blocks=32, L_max=L, N_max=N)
    try:
        load_weights(d, W)
        sig, ts = qi.flow_sigmas(40, N)
        t = _t(ts, 0)
        txt_np = synth.txt_feats(case)
        img_np = synth.img_tokens(case)
        txt, img = f32_tensor(txt_np), f32_tensor(img_np)
        (tc, tsn, ic, isn), (otc, ots, oic, ois) = _tables(L, h, w)
        # image positions are centred: rows and columns reach -64..63
        assert oic.shape == (N, 64)
        cos, sin = np.concatenate([otc, oic]), np.concatenate([ots, ois])
        tr = Tracer(qi, d, R)
        run = lambda: d.step(img, txt, t, tc, tsn, ic, isn)
        rows_txt, rows_img = _sample_rows(L, N, seed=41)
        rows = np.concatenate([rows_txt, L + rows_img])
        mods = odit.row_mods(odit.modulation(W.glob, np.float32(t)), odit.modulation(W.glob, 0.0), L, R)
        for b in (0, 31):
            a_, b_ = tr.around(b, run)
            _check_block(W, b, a_, b_[rows], mods, L, cos, sin, rows, f"2048^2 block {b}")
        _check_embed(W, tr.at(0, run), img_np, txt_np, rows_txt, rows_img, L, "2048^2 embedding")
        x_fin = tr.at(32, run)
        rb = range_buffer(d)
        d.set_range_probe(rb)
        vel = run().clone()
        d.set_range_probe(None)
        check_ranges(rb.cpu().numpy(), "2048^2 joint step")
        _check_head(W, x_fin[L:], vel.cpu().numpy(), rows_img, "2048^2 head")
        cached = d.step_cached(img, L, t, ic, isn)
        d.check()
        assert np.array_equal(vel.cpu().numpy(), cached.cpu().numpy())
        assert np.isfinite(vel.cpu().numpy()).all()
    finally:
        d.close()
