"""Benchmark: Qwen-Image-2.1 DiT sampler steps at 1024^2 (N = 4096 image tokens, L = 407).

One bench step = one FlowMatch Euler step of the 40-step loop: a DiT pass through
all 32 blocks (the first step of every image is the joint pass that captures the
text K/V; the other 39 run the image rows over the stored text K/V) followed by the
Euler update. K timed steps run images back to back from step 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). Under torchrun each rank runs an independent
replica on its own GPU (the step has no exchange between images): weak scaling.
The reference arm times the CPU oracle on this host's cores on a bounded sample
(per bench step, 512 image rows of one 1024^2 block; 256 such slices make a step).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "DiT steps/s at 1024² (N=4096,L=407); achieved bf16 TFLOPS vs tensor peak"
CASE = synth.LOOP_1024
STEPS_PER_IMAGE = 40
H = W_ = 64
N = H * W_
L = CASE.L
HIDDEN, FFN, BLOCKS = 4096, 12288, 32
GU_STRIDE = 4                              # gate/up GEMM timed in blocks 0, 4, 8, ...
GU_BLOCKS = len(range(0, BLOCKS, GU_STRIDE))


def step_flops(joint: bool) -> int:
    """Algorithmic FLOPs of one DiT pass (GEMMs + attention), as in the oracle's accounting."""
    R = L + N if joint else N
    gemm = 2 * R * (4 * HIDDEN * HIDDEN + 3 * HIDDEN * FFN)
    att = N * (N + L) * 4 * HIDDEN + (L * (L + 1) // 2 * 4 * HIDDEN if joint else 0)
    return BLOCKS * (gemm + att)


def gateup_flops(joint: bool) -> int:
    R = L + N if joint else N
    return 2 * R * HIDDEN * (2 * FFN)


def launches_per_step(joint: bool) -> int:
    # timestep embed + 3 GEMVs, image projection (+ text pre-norm + text GEMM),
    # 5 kernels per block, output head, Euler update
    return 4 + 1 + (2 if joint else 0) + 5 * BLOCKS + 1 + 1


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["bf16_tflops"], p.get("bf16_tflops_sustained"), p["hbm_gbs"], "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


class Clocks:
    """nvidia-smi sampling (200 ms) during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        time.sleep(0.3)
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.flush()
        rows = []
        with open(self.f.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ----------------------------------------------------------------------------- oracle (CPU)


SAMPLE_ROWS = 512
SAMPLES_PER_STEP = (N // SAMPLE_ROWS) * BLOCKS  # oracle slices that make one image-only step


def oracle_block_sample(samples: int, seed: int = CASE.seed):
    """Time the oracle on `samples` slices of an image-only 1024^2 block.

    A slice is 512 image rows of one block: their QKV projection and RoPE,
    attention over all L + N keys (image rows see every key, so the oracle's
    plain SDPA applies) and the out-projection and SwiGLU MLP. The block's K/V
    over all rows are computed once beforehand, as the sampler would hold them.
    One image-only step is SAMPLES_PER_STEP such slices. Returns seconds per slice.
    """
    from oracle import attention as oatt
    from oracle import dit as odit
    from oracle import rope as orope
    Wt = synth.Weights(seed=seed, nblocks=1)
    bw = Wt.block(0)
    x = synth.input_f32(seed, 90, (L + N, HIDDEN))
    tc, ts, ic, is_ = orope.token_tables(L, H, W_)
    cos, sin = np.concatenate([tc, ic]), np.concatenate([ts, is_])
    mods = odit.row_mods(odit.modulation(Wt.glob, 0.5), odit.modulation(Wt.glob, 0.0), L, L + N)
    s1, g1, s2, g2 = odit.mod_chunks(mods)
    _, k, v = odit.block_qkv(bw, x, s1, cos, sin, 32)
    times = []
    for i in range(samples):
        lo = L + (i * SAMPLE_ROWS) % N
        rows = slice(lo, lo + SAMPLE_ROWS)
        t0 = time.perf_counter()
        q, _, _ = odit.block_qkv(bw, x[rows], s1[rows], cos[rows], sin[rows], 32)
        o = oatt.sdpa(q, k, v, causal=False).reshape(SAMPLE_ROWS, HIDDEN)
        odit.block_after_attention(bw, x[rows], o, g1[rows], s2[rows], g2[rows])
        times.append(time.perf_counter() - t0)
    return times


def step_mix(steps: int):
    """(joint, image-only) steps among `steps` sampler steps of back-to-back 40-step images."""
    njoint = sum(1 for i in range(steps) if i % STEPS_PER_IMAGE == 0)
    return njoint, steps - njoint


def arm_config(world: int, steps: int) -> dict:
    """The workload both arms report."""
    njoint, nimg = step_mix(steps)
    return {"workload": "1024^2 sampler steps: N=4096 image tokens, L=407 text rows, 32 blocks, "
                        "40-step images back to back (step 0 joint + text K/V capture, 39 image-only)",
            "global_batch": world, "seq_len": L + N, "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2: 14.2 GB of weights stream through every step",
            "joint_steps": njoint, "image_only_steps": nimg}


def cores_used() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count() or 1


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's figure: the replicas run at once and the job ends with the last."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    nsamp = args.warmup + args.steps
    times = oracle_block_sample(nsamp)
    timed = times[args.warmup:]
    image_step = float(np.mean(timed)) * SAMPLES_PER_STEP
    # the same step mix as the GPU arm: a joint step costs its algorithmic FLOPs' share more
    njoint, nimg = step_mix(args.steps)
    per_step = image_step * (njoint * step_flops(True) + nimg * step_flops(False)) / (args.steps * step_flops(False))
    value = 1.0 / per_step
    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": arm_config(world, args.steps),
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "steps/s", "cores": cores_used(), "kind": "oracle",
                         "sample": f"per bench step one oracle slice (numpy fp32): 512 image rows of one "
                                   f"block with precomputed K/V; an image-only step is {SAMPLES_PER_STEP} slices, "
                                   f"a joint step that times its algorithmic FLOPs over an image-only step's; "
                                   f"{len(timed)} timed slices"},
        "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm


def gpu_weights(dit, seed, device):
    """Random-init bf16 weights drawn on the device (seeded), N(0, 0.02)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)

    def t(*shape):
        return (torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * 0.02).to(torch.bfloat16)

    d = synth.FULL
    dit.load_global({name: t(*shp(d)) for name, shp, _ in synth.GLOBAL_TENSORS})
    for b in range(BLOCKS):
        dit.load_block(b, {name: t(*shp(d)) for name, shp, _ in synth.BLOCK_TENSORS})
    torch.cuda.synchronize()


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import diffusion_transformer_text_gb300 as qi

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    qi.build()
    stream = torch.cuda.current_stream()

    dit = qi.DiT(blocks=BLOCKS, L_max=L, N_max=N, device=local_rank, kv_slots=2, mxfp8=True)
    gpu_weights(dit, CASE.seed * 1000 + rank, dev)

    sig, ts = qi.flow_sigmas(STEPS_PER_IMAGE, N)
    tvals = [float(np.float32(ts[i]) / np.float32(1000.0)) for i in range(STEPS_PER_IMAGE)]
    tc, tsn, ic, isn = qi.rope_tables(L, H, W_)
    g = torch.Generator(device=dev)
    g.manual_seed(1234 + rank)
    txt = torch.randn(L, HIDDEN, generator=g, device=dev)
    z = torch.randn(64, H, W_, generator=g, device=dev)
    x = qi.pack_noise(z)
    x0 = x.clone()
    vel = torch.empty(N, 64, device=dev)

    def sampler_step(i):
        k = i % STEPS_PER_IMAGE
        if k == 0:
            x.copy_(x0)
            dit.step(x, txt, tvals[0], tc, tsn, ic, isn, vel=vel)
        else:
            dit.step_cached(x, L, tvals[k], ic, isn, vel=vel)
        qi.euler_update(x, vel, float(sig[k]), float(sig[k + 1]))

    def barrier():
        if world > 1:
            dist.barrier()

    # warm-up (its own image), then the timed images start at step 0
    for i in range(args.warmup):
        sampler_step(i)
    torch.cuda.synchronize()
    dit.check()

    try:  # nvidia-smi ignores CUDA_VISIBLE_DEVICES: address the GPU by UUID
        uuid = str(torch.cuda.get_device_properties(local_rank).uuid)
        gpu_id = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
    except Exception:
        gpu_id = str(local_rank)
    clocks = Clocks(gpu_id)
    # CUDA events around the dominant kernel only (its roofline figure), in every
    # GU_STRIDE-th block: an event between two kernels also stops the second from
    # starting its set-up under the first, so events around every kernel class cost
    # ~1 % of a pass; the per-class split comes from a separate pass below
    dit.profile(True, classes=["gateup_gemm"], block_stride=GU_STRIDE)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        sampler_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier()
    prof = dit.profile_read()
    dit.profile(False)
    dit.check()
    ms = max_over_ranks(e0.elapsed_time(e1), world)

    njoint, nimg = step_mix(args.steps)
    flops = njoint * step_flops(True) + nimg * step_flops(False)
    value = world * args.steps / (ms / 1e3)
    tflops = world * flops / (ms / 1e3) / 1e12

    BREAKDOWN_STEPS = 10

    def breakdown():
        """Per-step device time of each kernel class over BREAKDOWN_STEPS sampler steps
        (1 joint + image-only) with every class timed by CUDA events."""
        x.copy_(x0)
        dit.profile(True)
        for i in range(BREAKDOWN_STEPS):
            sampler_step(i)
        torch.cuda.synchronize()
        kp = dit.profile_read()
        dit.profile(False)
        dit.check()
        return {k: v[0] / BREAKDOWN_STEPS for k, v in kp.items()}

    kernel_ms = breakdown()

    # ---- classifier-free guidance (second K/V slot): a 9-token negative prompt (the
    # host contract's empty-prompt template), guidance 2.5; 1 joint + CFG_STEPS - 1 cached
    CFG_STEPS, L_NEG, GUIDE = 10, 9, 2.5
    neg_txt = torch.randn(L_NEG, HIDDEN, generator=g, device=dev)
    ntc, nts, nic, nis = qi.rope_tables(L_NEG, H, W_)
    pos_p = dict(feats=txt, L=L, txt_cos=tc, txt_sin=tsn, img_cos=ic, img_sin=isn)
    neg_p = dict(feats=neg_txt, L=L_NEG, txt_cos=ntc, txt_sin=nts, img_cos=nic, img_sin=nis)
    x.copy_(x0)
    dit.step_cfg(x, tvals[0], GUIDE, pos_p, neg_p, vel=vel)  # warm-up
    torch.cuda.synchronize()
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for i in range(CFG_STEPS):
        dit.step_cfg(x, tvals[i], GUIDE, pos_p, neg_p, use_cache=i > 0, vel=vel)
        qi.euler_update(x, vel, float(sig[i]), float(sig[i + 1]))
    c1.record(stream)
    torch.cuda.synchronize()
    dit.check()
    cfg_ms = c0.elapsed_time(c1) / CFG_STEPS

    # ---- DPM++ 2M sampler: the same DiT passes with the second-order multistep update
    DPM_STEPS = 10
    d_prev = torch.empty_like(x)
    x.copy_(x0)
    torch.cuda.synchronize()
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for i in range(DPM_STEPS):
        if i == 0:
            dit.step(x, txt, tvals[0], tc, tsn, ic, isn, vel=vel)
        else:
            dit.step_cached(x, L, tvals[i], ic, isn, vel=vel)
        qi.dpmpp2m_update(x, vel, d_prev, sig, i)
    p1.record(stream)
    torch.cuda.synchronize()
    dit.check()
    dpm_ms = p0.elapsed_time(p1) / DPM_STEPS

    # ---- first-block cache ("Fast mode") at the pages' threshold 0.08, Euler loop
    FB_STEPS, FB_THR = 10, 0.08
    x.copy_(x0)
    torch.cuda.synchronize()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    skips, rels = 0, []
    f0.record(stream)
    for i in range(FB_STEPS):
        _, rel, sk = dit.step_fbcache(x, txt, L, tvals[i], tc, tsn, ic, isn, FB_THR, use_cache=i > 0, vel=vel)
        skips += sk
        rels.append(rel)
        qi.euler_update(x, vel, float(sig[i]), float(sig[i + 1]))
    f1.record(stream)
    torch.cuda.synchronize()
    fb_ms = f0.elapsed_time(f1) / FB_STEPS
    # a call that skips blocks 1..31: the same input again has zero change
    SKIP_REPS = 5
    dit.step_fbcache(x, txt, L, tvals[FB_STEPS], tc, tsn, ic, isn, FB_THR, use_cache=True, vel=vel)
    torch.cuda.synchronize()
    f0.record(stream)
    skipped_all = True
    for i in range(SKIP_REPS):
        _, rel, sk = dit.step_fbcache(x, txt, L, tvals[FB_STEPS], tc, tsn, ic, isn, FB_THR, use_cache=True, vel=vel)
        skipped_all &= sk
    f1.record(stream)
    torch.cuda.synchronize()
    dit.check()
    skip_ms = f0.elapsed_time(f1) / SKIP_REPS

    # ---- MXFP8 block GEMMs: block-scaled E4M3 weights and activations (a separate mode)
    MX_STEPS = 10
    dit.set_mxfp8(True)
    x.copy_(x0)
    dit.step(x, txt, tvals[0], tc, tsn, ic, isn, vel=vel)  # warm-up
    torch.cuda.synchronize()
    m0 = torch.cuda.Event(enable_timing=True)
    m1 = torch.cuda.Event(enable_timing=True)
    x.copy_(x0)
    dit.profile(True, classes=["gateup_gemm"], block_stride=GU_STRIDE)
    m0.record(stream)
    for i in range(MX_STEPS):
        if i == 0:
            dit.step(x, txt, tvals[0], tc, tsn, ic, isn, vel=vel)
        else:
            dit.step_cached(x, L, tvals[i], ic, isn, vel=vel)
        qi.euler_update(x, vel, float(sig[i]), float(sig[i + 1]))
    m1.record(stream)
    torch.cuda.synchronize()
    mx_prof = dit.profile_read()
    dit.profile(False)
    dit.check()
    mx_kernel_ms = breakdown()
    dit.set_mxfp8(False)
    mx_ms = m0.elapsed_time(m1) / MX_STEPS
    mx_flops = (step_flops(True) + (MX_STEPS - 1) * step_flops(False)) / MX_STEPS
    mx_gu_ms, _ = mx_prof["gateup_gemm"]
    mx_gu_flops = GU_BLOCKS * (gateup_flops(True) + (MX_STEPS - 1) * gateup_flops(False))

    # ---- end to end through the public API with host buffers
    xh = torch.empty(N, 64, dtype=torch.float32).pin_memory()
    xh.copy_(x0.cpu())
    txth = txt.cpu().pin_memory()
    tabs_h = [t.cpu().pin_memory() for t in (tc, tsn, ic, isn)]
    txt_d = torch.empty_like(txt)
    tabs_d = [torch.empty_like(t) for t in (tc, tsn, ic, isn)]

    def e2e_step(i):
        k = i % STEPS_PER_IMAGE
        x.copy_(xh, non_blocking=True)
        if k == 0:
            txt_d.copy_(txth, non_blocking=True)
            for d_, h_ in zip(tabs_d, tabs_h):
                d_.copy_(h_, non_blocking=True)
            dit.step(x, txt_d, tvals[0], *tabs_d, vel=vel)
        else:
            tabs_d[2].copy_(tabs_h[2], non_blocking=True)
            tabs_d[3].copy_(tabs_h[3], non_blocking=True)
            dit.step_cached(x, L, tvals[k], tabs_d[2], tabs_d[3], vel=vel)
        qi.euler_update(x, vel, float(sig[k]), float(sig[k + 1]))
        xh.copy_(x, non_blocking=True)

    e2e_steps = args.steps
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    h2d = (N * 64 * 4 + 2 * N * 64 * 4) * e2e_steps + njoint * (L * HIDDEN * 4 + 2 * L * 64 * 4)
    d2h = N * 64 * 4 * e2e_steps

    peak_b, peak_s, hbm, peak_kind = peaks()
    gu_ms, gu_n = prof["gateup_gemm"]
    gu_flops = GU_BLOCKS * (njoint * gateup_flops(True) + nimg * gateup_flops(False))
    gu_tflops = gu_flops / (gu_ms / 1e3) / 1e12 if gu_ms > 0 else None
    # dram read + write bytes per gate/up launch from the last ncu capture of this kernel
    traffic = None
    try:
        with open(os.path.join(ROOT, "profiles", "traffic_gateup_gemm.txt")) as f:
            traffic = float(f.read().split()[0])
    except Exception:
        pass

    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16",
        "dtype_note": "tensor-core products on fp16 operands (the bf16 weights convert exactly) with fp32 "
                      "accumulation; fp32 residual stream, norms, modulation and softmax statistics",
        "data": "synthetic",
        "config": arm_config(world, args.steps),
        "achieved_tflops": tflops,
        "tflops_frac_of_peak": tflops / world / peak_b,
        "tflops_frac_of_sustained_peak": tflops / world / peak_s,
        "gpu_launches": njoint * launches_per_step(True) + nimg * launches_per_step(False),
        "roofline": {"kernel": "gate/up GEMM + SwiGLU epilogue (tcgen05)", "bound": "tensor",
                     "achieved": gu_tflops, "peak": peak_s, "unit": "TFLOP/s",
                     "frac": (gu_tflops / peak_s) if gu_tflops else None, "traffic": traffic,
                     "peak_kind": f"{peak_kind} bf16 sustained (the kernel runs inside a seconds-long loop)",
                     "frac_of_burst": (gu_tflops / peak_b) if gu_tflops else None, "launches": gu_n,
                     "avg_launch_ms": gu_ms / gu_n if gu_n else None},
        "kernel_ms_per_step": kernel_ms,
        "kernel_ms_note": f"separate {BREAKDOWN_STEPS}-step pass (1 joint + image-only) with every kernel class "
                          "timed by CUDA events; the timed steps above carry events around the gate/up GEMM only",
        "e2e": {"value": world * e2e_steps / e2e_s, "unit": "steps/s", "h2d_bytes_per_step": h2d / e2e_steps,
                "d2h_bytes_per_step": d2h / e2e_steps},
        "clocks": clk,
        "cfg": {"steps_per_s": world * 1e3 / cfg_ms, "ms_per_step": cfg_ms, "guidance": GUIDE, "neg_tokens": L_NEG,
                "steps": CFG_STEPS, "note": "step 0: two joint passes (each prompt captures its K/V slot); "
                                            f"{CFG_STEPS - 1} image-only steps: one pass of 2N rows (batch 2)"},
        "dpmpp2m": {"steps_per_s": world * 1e3 / dpm_ms, "ms_per_step": dpm_ms, "steps": DPM_STEPS,
                    "note": "DPM++ 2M update in place of Euler, 1 joint + image-only passes"},
        "fbcache": {"threshold": FB_THR, "steps": FB_STEPS, "skipped": skips, "ms_per_step": fb_ms,
                    "steps_per_s": world * 1e3 / fb_ms, "rel_change": [None if r == float("inf") else r for r in rels],
                    "skipped_call_ms": skip_ms if skipped_all else None,
                    "note": "Euler loop under the first-block cache; random-init weights change block 0's "
                            "residual by ~0.9 per step, so nothing is skipped there; skipped_call_ms times a "
                            "call that skips blocks 1..31 (same input again)"},
    }
    fp8_peak = 2.0 * peak_b  # the recipe's nominal fp8 / bf16 ratio (4.5 / 2.25) on the measured bf16 burst
    line["mxfp8"] = {
        "steps_per_s": world * 1e3 / mx_ms, "ms_per_step": mx_ms, "steps": MX_STEPS,
        "achieved_tflops": mx_flops / (mx_ms / 1e3) / 1e12,
        "gateup_tflops": mx_gu_flops / (mx_gu_ms / 1e3) / 1e12 if mx_gu_ms > 0 else None,
        "fp8_peak_tflops": fp8_peak, "peak_kind": f"{peak_kind} bf16 burst x 2 (nominal fp8/bf16 ratio)",
        "kernel_ms_per_step": mx_kernel_ms,
        "note": "block GEMMs on MXFP8 (E4M3, UE8M0 scale per 32); activations quantised by a separate "
                "kernel before each GEMM (inside the GEMM classes of kernel_ms_per_step, measured in a separate "
                f"{BREAKDOWN_STEPS}-step pass); 1 joint + image-only"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        times = oracle_block_sample(9)
        image_step = float(np.mean(times[1:])) * SAMPLES_PER_STEP
        per_step = image_step * flops / (args.steps * step_flops(False))  # the timed steps' joint / image-only mix
        line["cpu_baseline"] = {"value": 1.0 / per_step, "unit": "steps/s", "cores": cores_used(),
                                "kind": "oracle",
                                "sample": f"8 timed oracle slices (numpy fp32, 512 image rows of one 1024^2 block "
                                          f"each, K/V precomputed), scaled by {SAMPLES_PER_STEP} slices per "
                                          f"image-only step and by algorithmic FLOPs to the timed steps' mix"}
    dit.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    rc = run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())
