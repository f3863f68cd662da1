"""bench.py's multi-process path on the CPU: two `gloo` ranks (127.0.0.1 rendezvous).

The benchmark runs replicas (one independent call per GPU), so the only cross-rank steps are
the rendezvous, the max over ranks of the timed interval, and rank 0 alone printing the JSON
line; these run here without a GPU.
"""
import json
import os
import socket
import subprocess
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    # every rank reports its own interval; all of them must come back with the largest
    got = bench.barrier_max(10.0 * (rank + 1), w)
    out.put((rank, got, dist.get_backend()))
    dist.destroy_process_group()


def test_barrier_max_over_two_gloo_ranks():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert res == [(0, 20.0, "gloo"), (1, 20.0, "gloo")]


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.barrier_max(3.5, 1) == 3.5


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus",
           "2", "--workload", "clip_n256", "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    t0 = time.perf_counter()
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    wall_ms = 1000 * (time.perf_counter() - t0)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] == 0
    assert d["unit"] == d["e2e"]["unit"] == d["cpu_baseline"]["unit"] == "pairs/s"
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["config"]["workload"] == "clip_n256"
    # the same workload description as the native arm's line (both come from run_config)
    sys.path.insert(0, ROOT)
    import bench
    from contrastive_embedding_loss_gb300 import synth

    kind, A16, B16, scale, bias = synth.workload("clip_n256")
    args = type("Args", (), {"workload": "clip_n256"})()
    assert d["config"] == json.loads(json.dumps(bench.run_config(args, kind, A16, B16, scale, bias, 2)))
    # its step time is the time of the step as run (a sub-batch), which fits inside the run
    assert 0 < d["ms_per_step"] * (d["steps"] + d["warmup"]) <= wall_ms
    assert d["ms_per_step_full_batch"] >= d["ms_per_step"]


@pytest.mark.parametrize("impl", ["native"])
def test_native_arm_fails_loudly_without_a_gpu(impl):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", impl, "--steps", "1", "--warmup",
                        "0", "--workload", "clip_n256", "--no-cpu-baseline"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode != 0  # no CUDA path, and no silent CPU fallback
