"""The N > 1 bench path on the CPU: replicas only, joined by a gloo process group
(world size 2 on 127.0.0.1). The timed figure is the slowest rank's, and under a
torchrun-style launch only rank 0 of the reference arm prints."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, init_method=f"tcp://127.0.0.1:{port}")
    import bench
    q.put((rank, bench.max_over_ranks(10.0 + 5.0 * rank, world)))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 15.0, 1: 15.0}


def test_single_rank_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5


@pytest.mark.slow
def test_reference_arm_prints_on_rank_0_only():
    """The reference arm under WORLD_SIZE=2: rank 1 exits 0 silently, rank 0 prints one line."""
    outs = []
    for rank in (1, 0):
        env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank))
        r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        outs.append(r.stdout.strip())
    assert outs[0] == ""
    line = json.loads(outs[1].splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    # the same workload description as the GPU arm's line
    sys.path.insert(0, ROOT)
    import bench
    assert line["config"] == bench.arm_config(2, 1)
    assert line["e2e"]["value"] == line["value"] and line["cpu_baseline"]["value"] == line["value"]


def test_step_mix():
    """Back-to-back 40-step images: step 0 of each image is the joint pass."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.step_mix(40) == (1, 39)
    assert bench.step_mix(41) == (2, 39)
    assert bench.step_mix(1) == (1, 0)
    cfg = bench.arm_config(4, 80)
    assert cfg["joint_steps"] == 2 and cfg["image_only_steps"] == 78 and cfg["global_batch"] == 4


def test_bench_flop_model_matches_the_oracle_accounting():
    """The bench's per-pass and per-kernel-class FLOPs equal the oracle's step model on every workload."""
    import bench
    from oracle import dit as odit
    for case in (synth_cases()):
        for joint in (True, False):
            R = case.L + case.N if joint else case.N
            want = odit.step_flops(R, case.N, case.L, joint)
            assert bench.pass_flops(case.L, case.N, joint) == want
            assert sum(bench.class_flops(case.L, case.N, joint).values()) == want
    # 598 rows at 384^2 with a 22-token prompt: about 8.5 TFLOP (MLX page, "Where the time goes")
    assert abs(bench.pass_flops(22, 576, True) / 1e12 - 8.5) < 0.05


def test_bench_clock_normalised_fraction():
    import bench
    # the same TFLOP/s per MHz as the peak is a fraction of 1, whatever the two clocks
    assert abs(bench.frac_at_clock(1000.0, 1500.0, 1200.0, 1800.0) - 1.0) < 1e-12
    assert abs(bench.frac_at_clock(1715.5, 1650.0, 1741.2, 1492.0) - 0.8909) < 1e-3
    assert bench.frac_at_clock(1000.0, None, 1200.0, 1800.0) is None


def synth_cases():
    import synth
    return (synth.STEP_256, synth.STEP_384_L22, synth.STEP_384_L494, synth.LOOP_1024, synth.STEP_2048)
